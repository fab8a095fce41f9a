// The verify step of speculative decoding ("5. Core modules" 5.6): n drafts of one session as the rows of
// one decode step, or through the chunk path, and the truncation to the accepted prefix.
#include "engine.h"

namespace mag {

// Verify step on the decode kernels: the n tokens are the n rows of a decode step of one session at
// positions len .. len + n - 1, with their keys and values stored between the QKV projection and attention.
static mag_status verify_on_step(mag_ctx* c, int32_t sid, int32_t n, const void* in, void* out) {
  mag_status st = poll_capture(c);
  if (st != MAG_OK) return st;
  if (sid < 0 || sid >= (int)c->sessions.size() || !c->sessions[sid].open)
    return fail(c, MAG_ERR_INVALID_ARG, "verify_tokens: session %d is not open", sid);
  if (!all_loaded(c)) return fail(c, MAG_ERR_NOT_LOADED, "verify_tokens: not every weight is loaded");
  Session& s = c->sessions[sid];
  if ((int64_t)s.len + n > c->cfg.max_context)
    return fail(c, MAG_ERR_CONTEXT_FULL, "verify_tokens: %d + %d tokens exceed max_context %d", s.len, n,
                c->cfg.max_context);
  // n <= 16 tokens reach at most one block past the session's last one
  const int nb_old = (s.len + 15) / 16, nb_new = (s.len + n + 15) / 16;
  st = reserve_blocks(c, "verify_tokens", nb_new - nb_old);
  if (st != MAG_OK) return st;
  const int slot = c->ring_pos;
  CUDA_TRY(c, cudaEventSynchronize(c->ring_ev[slot]));
  StepArgs& a = c->h_ring[slot];
  memset(&a, 0, sizeof a);
  a.batch = n;
  for (int b = 0; b < n; ++b) {
    a.sess[b] = sid;
    a.pos[b] = s.len + b;
  }
  c->step_max_len = s.len + n;
  for (int i = nb_old; i < nb_new; ++i) {
    const int blk = c->kv.pop();
    s.table.push_back(blk);
    a.upd_sess[a.n_upd] = sid;
    a.upd_idx[a.n_upd] = i;
    a.upd_blk[a.n_upd] = blk;
    ++a.n_upd;
  }
  for (int b = 0; b < n; ++b) a.blk[b] = s.table[(s.len + b) / 16];
  a.hidden_in = (const __half*)in;
  a.out = out;
  CUDA_TRY(c, cudaMemcpyAsync(c->d_args, &a, sizeof a, cudaMemcpyHostToDevice, c->stream));
  CUDA_TRY(c, cudaEventRecord(c->ring_ev[slot], c->stream));
  c->ring_pos = (slot + 1) % kRing;
  int32_t lens[MAG_MAX_BATCH];
  for (int b = 0; b < n; ++b) lens[b] = s.len + b + 1;
  st = stats_begin(c, 1, n, n, lens, n);
  if (st != MAG_OK) return st;
  st = launch_step(c, n, true);
  if (st != MAG_OK) return st;
  st = stats_end(c);
  if (st != MAG_OK) return st;
  s.len += n;
  adapt_after_step(c, n, lens);
  return pool_trim(c);
}

}  // namespace mag

extern "C" {

mag_status mag_verify_tokens(mag_ctx* c, int32_t sid, int32_t n_tokens, const void* hidden_in, void* out) {
  if (!c) return MAG_ERR_INVALID_ARG;
  if (!hidden_in || !out) return fail(c, MAG_ERR_INVALID_ARG, "verify_tokens: null buffer");
  // up to max_batch tokens on the decode kernels (weights read once for all rows); beyond that, up to
  // kPipeMaxBatch tokens through the prefill chunk path when the context has one
  if (n_tokens >= 1 && n_tokens <= c->B_max) return verify_on_step(c, sid, n_tokens, hidden_in, out);
  const int chunk_max = std::min(kPipeMaxBatch, c->cfg.max_chunk);
  if (n_tokens >= 1 && n_tokens <= chunk_max)
    return run_chunk(c, "verify_tokens", 1, &sid, &n_tokens, hidden_in, out, true);
  return fail(c, MAG_ERR_INVALID_ARG, "verify_tokens: %d tokens not in 1..%d", n_tokens,
              std::max(c->B_max, chunk_max));
}

mag_status mag_session_truncate(mag_ctx* c, int32_t sid, int32_t length) {
  if (!c) return MAG_ERR_INVALID_ARG;
  if (sid < 0 || sid >= (int)c->sessions.size() || !c->sessions[sid].open)
    return fail(c, MAG_ERR_INVALID_ARG, "session_truncate: session %d is not open", sid);
  Session& s = c->sessions[sid];
  if (length < 0 || length > s.len)
    return fail(c, MAG_ERR_INVALID_ARG, "session_truncate: length %d not in 0..%d", length, s.len);
  // blocks wholly past the new length go back to the pool; the device table keeps stale entries past
  // the length, which nothing reads, and a later append writes the new ids before they are used
  const size_t nb = (size_t)(length + 15) / 16;
  while (s.table.size() > nb) {
    c->kv.push(s.table.back());
    s.table.pop_back();
  }
  s.len = length;
  return pool_trim(c);
}

}  // extern "C"
