// The decode step: its launches (one CUDA graph per batch size, attention shape and step kind), the step
// arguments' upload, the adaptive plans and their background capture.
#include "engine.h"

namespace mag {

// Enqueue the whole decode step for batch B (captured into a graph or run eagerly).
// The decode step's launches. With `verify` the B rows are B consecutive new tokens of one session: their
// keys and values go into the pool in one store kernel after the QKV projection, and attention reads them
// there (row b causally up to its own position) instead of each row appending its own.
// `splits` is the attention split count of the plan in use; `st` the stream the launches go to (the
// context's, or a capture stream). With `resid_dump` (eager debug steps only) the fp32 residual of the B rows
// is copied there after the step prologue and after every layer: [L+1][B][D].
cudaError_t record_step(mag_ctx* c, int B, int* n_launch, Profiler* prof, bool verify, int splits, bool wide,
                        cudaStream_t st, float* resid_dump) {
  const bool pdl = !(c->cfg.flags & MAG_FLAG_NO_PDL) && !prof && !resid_dump;
  auto dump = [&](int row) {
    return resid_dump ? cudaMemcpyAsync(resid_dump + (size_t)row * B * c->D, c->r, (size_t)B * c->D * 4,
                                        cudaMemcpyDeviceToDevice, st)
                      : cudaSuccess;
  };
  Launch L0{st, false, n_launch};
  Launch L{st, pdl, n_launch};
  cudaError_t e;
  // every launch goes through MAG_RUN, which brackets it with events when profiling
#define MAG_RUN(kind, call)                                            \
  do {                                                                \
    if (prof && (e = prof->begin(st)) != cudaSuccess) return e;       \
    if ((e = (call)) != cudaSuccess) return e;                        \
    if (prof && (e = prof->end(st, (kind))) != cudaSuccess) return e; \
  } while (0)
  MAG_RUN(MAG_OP_STEP_BEGIN,
          launch_step_begin(L0, c->d_args, c->r, c->D, c->d_tables, c->table_stride, B, c->ss_part));
  if ((e = dump(0)) != cudaSuccess) return e;
  const PoolGeom pg = pool_geom(c);
  const int S = splits;
  const bool kv_by_qkv = !verify && c->cfg.kv_dtype == MAG_KV_FP16 && B <= kPipeMaxBatch;
  for (int l = 0; l < c->L; ++l) {
    const Proj* P = &c->proj[(size_t)l * 4];
    {  // RMSNorm + QKV + RoPE of q and k
      GemvArgs a = gemv_args(c, 0, P[0].tiles, c->R / 16, c->D, B);
      a.n_ss = l == 0 ? 1 : c->D / 16;  // the step prologue leaves one sum per token
      a.gamma = c->gamma1[l];
      a.out_h = c->qkv;
      a.ldo = c->R;
      a.head_dim = c->d;
      a.n_rot_heads = c->Hq + c->Hkv;
      a.rope_cos = c->d_cos;
      a.rope_sin = c->d_sin;
      // FP16 pool, decode rows on the pipelined GEMV: its epilogue also stores each row's key and value
      a.kv_store = kv_by_qkv ? 1 : 0;
      a.n_q_heads = c->Hq;
      a.layer = l;
      a.pool = pg;
      MAG_RUN(MAG_OP_QKV, launch_gemv(L, a, W_W4, XSRC_RESID, EPI_QKV));
    }
    if (verify) {  // the B tokens' k and v into the pool
      KvChunkArgs kc = {};
      kc.err = c->d_err;
      kc.qkv = c->qkv;
      kc.qkv_ld = c->R;
      kc.n_heads = c->Hq;
      kc.n_tok = B;
      kc.layer = l;
      kc.pool = pg;
      kc.step = c->d_args;
      MAG_RUN(MAG_OP_ATTENTION, launch_kv_store_chunk(L, kc));
    }
    {  // KV append + attention
      AttnArgs a = {};
      a.qkv = c->qkv;
      a.qkv_ld = c->R;
      a.o = c->o;
      a.ldo = c->Hq * c->d;
      a.n_heads = c->Hq;
      a.n_kv_heads = c->Hkv;
      a.head_dim = c->d;
      a.layer = l;
      a.pool = pg;
      a.step = c->d_args;
      a.stored = verify ? 1 : (kv_by_qkv ? 2 : 0);
      a.wide = wide;
      // more splits than one cluster holds: clusters of at most 8 (which co-schedule more readily than
      // clusters of 16), merged by the last block to finish
      const int cmax = wide ? c->attn_cluster_max_wide : c->attn_cluster_max;
      const int csz = S <= cmax ? cmax : std::min(cmax, 8);
      a.n_groups = std::min(kAttnMaxGroups, (S + csz - 1) / csz);
      a.n_split = std::min(csz, (S + a.n_groups - 1) / a.n_groups);
      a.part = c->attn_part;
      a.arrivals = c->attn_arrivals;
      a.err = c->d_err;
      a.trace = c->trace;
      MAG_RUN(MAG_OP_ATTENTION, launch_attention(L, a, B));
    }
    {  // O projection + residual
      GemvArgs a = gemv_args(c, 1, P[1].tiles, c->D / 16, c->Hq * c->d, B);
      a.x = c->o;
      a.ldx = c->Hq * c->d;
      MAG_RUN(MAG_OP_O, launch_gemv(L, a, W_W4, XSRC_F16, EPI_RESID));
    }
    {  // RMSNorm + gate-up + SwiGLU
      GemvArgs a = gemv_args(c, 2, P[2].tiles, c->F / 8, c->D, B);
      a.gamma = c->gamma2[l];
      a.out_h = c->act;
      a.ldo = c->F;
      MAG_RUN(MAG_OP_GATE_UP, launch_gemv(L, a, W_W4, XSRC_RESID, EPI_SWIGLU));
    }
    {  // down projection + residual
      GemvArgs a = gemv_args(c, 3, P[3].tiles, c->D / 16, c->F, B);
      a.x = c->act;
      a.ldx = c->F;
      MAG_RUN(MAG_OP_DOWN, launch_gemv(L, a, W_W4, XSRC_F16, EPI_RESID));
    }
    if ((e = dump(l + 1)) != cudaSuccess) return e;
  }
  if (c->V) {  // final RMSNorm + LM head
    GemvArgs a = gemv_args(c, 4, reinterpret_cast<const uint8_t*>(c->lm_head), c->V / 16, c->D, B);
    a.gamma = c->gamma_f;
    a.ldo = c->V;
    MAG_RUN(MAG_OP_LM_HEAD, launch_gemv(L, a, W_F16, XSRC_RESID, EPI_STORE_OUT));
  } else {
    MAG_RUN(MAG_OP_LM_HEAD, launch_final_hidden(L, c->d_args, c->r, c->D, B));
  }
  if (c->canary_band) {  // debug: the arena tensors' canary bands are intact
    if ((e = launch_arena_check(L, arena_check_args(c))) != cudaSuccess) return e;
  }
#undef MAG_RUN
  return cudaSuccess;
}

mag_status step_prepare(mag_ctx* c, int B, const int32_t* sids, StepArgs& a) {
  if (B < 1 || B > c->B_max) return fail(c, MAG_ERR_INVALID_ARG, "decode_step: batch %d not in 1..%d", B, c->B_max);
  if (!sids) return fail(c, MAG_ERR_INVALID_ARG, "decode_step: null session ids");
  if (!all_loaded(c)) return fail(c, MAG_ERR_NOT_LOADED, "decode_step: not every weight is loaded");
  int need = 0;
  for (int b = 0; b < B; ++b) {
    int s = sids[b];
    if (s < 0 || s >= (int)c->sessions.size() || !c->sessions[s].open)
      return fail(c, MAG_ERR_INVALID_ARG, "decode_step: session %d is not open", s);
    for (int j = 0; j < b; ++j)
      if (sids[j] == s) return fail(c, MAG_ERR_INVALID_ARG, "decode_step: session %d appears twice", s);
    if (c->sessions[s].len + 1 > c->cfg.max_context)
      return fail(c, MAG_ERR_CONTEXT_FULL, "decode_step: session %d is at max_context", s);
    if (c->sessions[s].len % 16 == 0) ++need;
  }
  mag_status st = reserve_blocks(c, "decode_step", need);
  if (st != MAG_OK) return st;
  a.batch = B;
  a.n_upd = 0;
  c->step_max_len = 0;
  for (int b = 0; b < B; ++b) {
    Session& s = c->sessions[sids[b]];
    a.sess[b] = sids[b];
    a.pos[b] = s.len;
    c->step_max_len = std::max(c->step_max_len, s.len + 1);
    if (s.len % 16 == 0) {
      int blk = c->kv.pop();
      s.table.push_back(blk);
      a.upd_sess[a.n_upd] = sids[b];
      a.upd_idx[a.n_upd] = s.len / 16;
      a.upd_blk[a.n_upd] = blk;
      ++a.n_upd;
    }
    a.blk[b] = s.table[s.len / 16];
  }
  return MAG_OK;
}

mag_status step_upload(mag_ctx* c, int B, const int32_t* sids, const void* in, void* out) {
  if (!in || !out) return fail(c, MAG_ERR_INVALID_ARG, "decode_step: null buffer");
  const int slot = c->ring_pos;
  CUDA_TRY(c, cudaEventSynchronize(c->ring_ev[slot]));
  StepArgs& a = c->h_ring[slot];
  memset(&a, 0, sizeof a);
  mag_status st = step_prepare(c, B, sids, a);
  if (st != MAG_OK) return st;
  a.hidden_in = (const __half*)in;
  a.out = out;
  CUDA_TRY(c, cudaMemcpyAsync(c->d_args, &a, sizeof a, cudaMemcpyHostToDevice, c->stream));
  CUDA_TRY(c, cudaEventRecord(c->ring_ev[slot], c->stream));
  c->ring_pos = (slot + 1) % kRing;
  return MAG_OK;
}

// Whether plan p runs the wide attention blocks.
bool plan_wide(const mag_ctx* c, int p) { return c->adapt.enable_adaptive && c->adapt.plan_wide[p]; }

// Attention split count of plan p at batch B: the plan's count (a single-session figure), capped at about
// 4 blocks per SM over the batch's (session, KV head) pairs; 0 = the context's default (at most one
// cluster).
int plan_splits(const mag_ctx* c, int p, int B) {
  const int s = c->adapt.enable_adaptive ? c->adapt.plan_splits[p] : 0;
  if (s == 0) return attn_splits(c, B, plan_wide(c, p));
  return std::max(1, std::min(s, 4 * c->n_sm / (B * c->Hkv)));
}

// Attention launch shape of the step being launched: the plan's with the adaptive runtime on; otherwise by
// the step's longest context, about 76 pool blocks per split (measured on GB300: 16 splits, one cluster, up
// to ~19k keys; 32 at ~39k; 64 at ~78k), so that long contexts keep enough warps streaming the pool.
AttnShape attn_shape(const mag_ctx* c, int B) {
  if (c->adapt.enable_adaptive) return {plan_splits(c, c->cur_plan, B), plan_wide(c, c->cur_plan), -1};
  const int nb = (c->step_max_len + 15) / 16, def = attn_splits(c, B);
  const int bk = nb <= 16 * 76 ? 0 : (nb <= 32 * 76 ? 1 : (nb <= 48 * 76 ? 2 : 3));
  const int s = bk == 0 ? def : std::max(def, std::min(16 * (bk + 1), 4 * c->n_sm / (B * c->Hkv)));
  return {s, false, bk};
}

// Capture and instantiate the step graph of (verify, plan p, batch B) on stream st: the context's
// stream, or the capture stream of a background switch.
cudaError_t capture_graph(mag_ctx* c, bool verify, int p, int B, cudaStream_t st,
                                 mag_ctx::StepGraph& out) {
  cudaGraph_t g = nullptr;
  int n = 0;
  cudaError_t e = cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) return e;
  e = record_step(c, B, &n, nullptr, verify, plan_splits(c, p, B), plan_wide(c, p), st);
  const cudaError_t e2 = cudaStreamEndCapture(st, &g);
  if (e == cudaSuccess) e = e2;
  if (e == cudaSuccess) e = cudaGraphInstantiate(&out.exec, g, 0);
  if (g) cudaGraphDestroy(g);
  if (e == cudaSuccess) out.launches = n;
  return e;
}

// A background capture that has finished: switch to its plan, or report why it failed.
mag_status poll_capture(mag_ctx* c) {
  const int s = c->cap_state.load(std::memory_order_acquire);
  if (s != 2 && s != 3) return MAG_OK;
  c->cap_thread.join();
  c->cap_state.store(0);
  const int p = c->pending_plan;
  c->pending_plan = -1;
  if (s == 3) return fail(c, MAG_ERR_CUDA, "capture of plan %d: %s", p, c->cap_err.c_str());
  c->cur_plan = p;
  ++c->switches;
  return MAG_OK;
}

// Wait for a background capture (before the graphs or the configuration change under it).
mag_status finish_capture(mag_ctx* c) {
  if (c->cap_thread.joinable()) c->cap_thread.join();
  return poll_capture(c);
}

// Switch to plan p: at once (its graphs are captured on first use by the step), or, with async_switch,
// after a background thread has captured p's graphs for every shape the current plan has captured.
void switch_plan(mag_ctx* c, int p) {
  std::vector<std::pair<int, int>> shapes;
  if (c->adapt.async_switch && !(c->cfg.flags & MAG_FLAG_NO_GRAPH))
    for (int v = 0; v < 2; ++v)
      for (int b = 1; b <= MAG_MAX_BATCH; ++b)
        if (c->graphs[v][c->cur_plan][b].exec && !c->graphs[v][p][b].exec) shapes.emplace_back(v, b);
  if (shapes.empty()) {
    c->cur_plan = p;
    ++c->switches;
    return;
  }
  c->pending_plan = p;
  c->cap_state.store(1);
  c->cap_thread = std::thread([c, p, shapes]() {
    cudaError_t e = cudaSetDevice(c->device);
    for (const auto& sh : shapes) {
      if (e != cudaSuccess) break;
      e = capture_graph(c, sh.first != 0, p, sh.second, c->cap_stream, c->graphs[sh.first][p][sh.second]);
    }
    if (e != cudaSuccess) c->cap_err = cudaGetErrorString(e);
    c->cap_state.store(e == cudaSuccess ? 2 : 3, std::memory_order_release);
  });
}

// Offer a finished step's rows (the context length each attended) to the load profile; on a recorded
// sample with the window full, update the hot pool target and pick the plan of the window's P90.
void adapt_after_step(mag_ctx* c, int B, const int32_t* lens) {
  if (!c->adapt.enable_adaptive) return;
  bool rec = false;
  for (int b = 0; b < B; ++b) rec |= c->profile->observe(lens[b]);
  if (!rec || !c->profile->full()) return;
  const int32_t p90 = c->profile->quantile(0.9);
  int open = 0;
  for (const Session& s : c->sessions) open += s.open;
  c->hot_blocks = hot_pool_blocks(p90, open, c->adapt.hot_pool_slack, 16);
  if (c->kv.elastic() &&
      c->kv.set_hot(c->hot_blocks, c->stream, [c](int64_t g) { return group_referenced(c, g); }) != MAG_OK)
    fail(c, MAG_ERR_OOM, "hot pool resize (kept the old size): %s", c->kv.err.c_str());
  if (c->adapt.force_plan >= 0 || c->pending_plan >= 0) return;
  const int want = plan_for(p90, c->adapt.plan_short_below, c->adapt.plan_long_above);
  if (want != c->cur_plan) switch_plan(c, want);
}

// Launches the step of B rows whose arguments were just uploaded: the captured graph of that shape
// under the plan in use (captured on first use), or the kernels one by one under MAG_FLAG_NO_GRAPH.
mag_status stats_begin(mag_ctx* c, int kind, int rows, int out_rows, const int32_t* keys, int n_keys_rows) {
  mag_step_stats& s = c->stats;
  const uint64_t per_token = mag_kv_bytes_per_token(&c->cfg);
  uint64_t kv = 0;
  int most = 0;
  for (int i = 0; i < n_keys_rows; ++i) {
    kv += (uint64_t)keys[i] * per_token;
    most = std::max(most, (int)keys[i]);
  }
  s.last_kind = kind;
  s.last_rows = rows;
  s.last_max_keys = most;
  s.last_bytes = (uint64_t)c->wbytes + kv + (uint64_t)rows * c->D * 2 + (uint64_t)out_rows * (c->V ? c->V : c->D) * 2;
  c->step_timed = (c->cfg.flags & MAG_FLAG_STEP_TIMING) != 0;
  if (c->step_timed) CUDA_TRY(c, cudaEventRecord(c->ev_step[0], c->stream));
  return MAG_OK;
}

mag_status stats_end(mag_ctx* c) {
  c->stats.steps += 1;
  c->stats.last_launches = c->last_launches;
  if (c->step_timed) CUDA_TRY(c, cudaEventRecord(c->ev_step[1], c->stream));
  return MAG_OK;
}

mag_status launch_step(mag_ctx* c, int B, bool verify) {
  const AttnShape sh = attn_shape(c, B);
  if (c->cfg.flags & MAG_FLAG_NO_GRAPH) {
    int n = 0;
    CUDA_TRY(c, record_step(c, B, &n, nullptr, verify, sh.splits, sh.wide, c->stream));
    c->last_launches = n;
    return MAG_OK;
  }
  mag_ctx::StepGraph& g = sh.bucket < 0 ? c->graphs[verify][c->cur_plan][B] : c->len_graphs[verify][sh.bucket][B];
  if (!g.exec && sh.bucket >= 0) {
    cudaGraph_t gr = nullptr;
    int n = 0;
    cudaError_t e = cudaStreamBeginCapture(c->stream, cudaStreamCaptureModeThreadLocal);
    if (e == cudaSuccess) {
      e = record_step(c, B, &n, nullptr, verify, sh.splits, sh.wide, c->stream);
      const cudaError_t e2 = cudaStreamEndCapture(c->stream, &gr);
      if (e == cudaSuccess) e = e2;
    }
    if (e == cudaSuccess) e = cudaGraphInstantiate(&g.exec, gr, 0);
    if (gr) cudaGraphDestroy(gr);
    if (e != cudaSuccess) return fail(c, MAG_ERR_CUDA, "step graph capture: %s", cudaGetErrorString(e));
    g.launches = n;
  }
  if (!g.exec) CUDA_TRY(c, capture_graph(c, verify, c->cur_plan, B, c->stream, g));
  CUDA_TRY(c, cudaGraphLaunch(g.exec, c->stream));
  c->last_launches = g.launches;
  return MAG_OK;
}

}  // namespace mag

extern "C" {

mag_status mag_decode_step(mag_ctx* c, int32_t B, const int32_t* sids, const void* in, void* out) {
  if (!c) return MAG_ERR_INVALID_ARG;
  mag_status st = poll_capture(c);
  if (st != MAG_OK) return st;
  st = step_upload(c, B, sids, in, out);
  if (st != MAG_OK) return st;
  int32_t lens[MAG_MAX_BATCH];
  for (int b = 0; b < B; ++b) lens[b] = c->sessions[sids[b]].len + 1;  // the keys row b attends
  st = stats_begin(c, 0, B, B, lens, B);
  if (st != MAG_OK) return st;
  st = launch_step(c, B, false);
  if (st != MAG_OK) return st;
  st = stats_end(c);
  if (st != MAG_OK) return st;
  for (int b = 0; b < B; ++b) ++c->sessions[sids[b]].len;
  adapt_after_step(c, B, lens);
  return pool_trim(c);
}

mag_status mag_debug_profile_step(mag_ctx* c, int32_t B, const int32_t* sids, const void* in, void* out,
                                  int32_t* kinds, float* ms, int32_t cap, int32_t* n_out) {
  if (!c || !n_out || cap < 0 || (cap && (!kinds || !ms))) return MAG_ERR_INVALID_ARG;
  mag_status st = step_upload(c, B, sids, in, out);
  if (st != MAG_OK) return st;
  Profiler prof;
  int n = 0;
  const AttnShape sh = attn_shape(c, B);
  CUDA_TRY(c, record_step(c, B, &n, &prof, false, sh.splits, sh.wide, c->stream));
  for (int b = 0; b < B; ++b) c->sessions[sids[b]].len += 1;
  CUDA_TRY(c, cudaStreamSynchronize(c->stream));
  *n_out = (int32_t)prof.kinds.size();
  for (int i = 0; i < (int)prof.kinds.size() && i < cap; ++i) {
    kinds[i] = prof.kinds[i];
    CUDA_TRY(c, cudaEventElapsedTime(&ms[i], prof.start[i], prof.stop[i]));
  }
  c->last_launches = n;
  return MAG_OK;
}

mag_status mag_debug_step_residuals(mag_ctx* c, int32_t B, const int32_t* sids, const void* in, void* out,
                                    void* resid) {
  if (!c) return MAG_ERR_INVALID_ARG;
  if (!resid) return fail(c, MAG_ERR_INVALID_ARG, "debug_step_residuals: null residual buffer");
  mag_status st = step_upload(c, B, sids, in, out);
  if (st != MAG_OK) return st;
  int n = 0;
  const AttnShape sh = attn_shape(c, B);
  CUDA_TRY(c, record_step(c, B, &n, nullptr, false, sh.splits, sh.wide, c->stream, static_cast<float*>(resid)));
  for (int b = 0; b < B; ++b) c->sessions[sids[b]].len += 1;
  CUDA_TRY(c, cudaStreamSynchronize(c->stream));
  c->last_launches = n;
  return check_err(c);
}

mag_status mag_debug_timeline(mag_ctx* c, int32_t B, const int32_t* sids, const void* in, void* out, void* recs,
                              int32_t cap, int32_t* n_out) {
  if (!c) return MAG_ERR_INVALID_ARG;
  if (!recs || cap < 0 || !n_out) return fail(c, MAG_ERR_INVALID_ARG, "debug_timeline: null buffer or count");
  mag_status st = finish_capture(c);
  if (st != MAG_OK) return st;
  if (!c->trace_n) {
    cudaError_t e = dev_malloc(&c->trace_n, sizeof(unsigned int));
    if (e != cudaSuccess) return fail(c, MAG_ERR_OOM, "debug_timeline: counter: %s", cudaGetErrorString(e));
  }
  st = step_upload(c, B, sids, in, out);
  if (st != MAG_OK) return st;
  CUDA_TRY(c, cudaMemsetAsync(c->trace_n, 0, sizeof(unsigned int), c->stream));
  c->trace = TraceBuf{static_cast<unsigned long long*>(recs), c->trace_n, (unsigned int)cap};
  int n = 0;
  const AttnShape sh = attn_shape(c, B);
  // the step's launches as the graph holds them (programmatic dependent launch included), but launched
  // one by one so that their arguments carry the record buffer
  const cudaError_t e = record_step(c, B, &n, nullptr, false, sh.splits, sh.wide, c->stream);
  c->trace = TraceBuf{};
  CUDA_TRY(c, e);
  for (int b = 0; b < B; ++b) c->sessions[sids[b]].len += 1;
  unsigned int got = 0;
  CUDA_TRY(c, cudaMemcpyAsync(&got, c->trace_n, sizeof got, cudaMemcpyDeviceToHost, c->stream));
  CUDA_TRY(c, cudaStreamSynchronize(c->stream));
  *n_out = (int32_t)std::min<unsigned int>(got, 0x7fffffffu);
  c->last_launches = n;
  return check_err(c);
}

mag_status mag_debug_set_wait_limit(mag_ctx* c, int64_t polls) {
  if (!c) return MAG_ERR_INVALID_ARG;
  mag_status st = finish_capture(c);
  if (st != MAG_OK) return st;
  const uint32_t v = polls < 0 ? kWaitPolls : (uint32_t)std::min<int64_t>(polls, 0xffffffffll);
  if (v == c->wait_limit) return MAG_OK;
  CUDA_TRY(c, cudaStreamSynchronize(c->stream));
  // captured graphs hold the old limit in their kernel arguments: capture again on next use
  for (auto& gv : c->len_graphs)
    for (auto& gp : gv)
      for (auto& g : gp)
        if (g.exec) {
          cudaGraphExecDestroy(g.exec);
          g = mag_ctx::StepGraph{};
        }
  for (auto& gv : c->graphs)
    for (auto& gp : gv)
      for (auto& g : gp)
        if (g.exec) {
          cudaGraphExecDestroy(g.exec);
          g = mag_ctx::StepGraph{};
        }
  c->wait_limit = v;
  return MAG_OK;
}

mag_status mag_decode_step_host(mag_ctx* c, int32_t B, const int32_t* sids, const void* in_host, void* out_host) {
  if (!c) return MAG_ERR_INVALID_ARG;
  if (!in_host || !out_host) return fail(c, MAG_ERR_INVALID_ARG, "decode_step_host: null buffer");
  if (B < 1 || B > c->B_max) return fail(c, MAG_ERR_INVALID_ARG, "decode_step_host: batch %d", B);
  const size_t in_b = (size_t)B * c->D * 2, out_b = (size_t)B * (c->V ? c->V : c->D) * 2;
  CUDA_TRY(c, cudaMemcpyAsync(c->d_in_stage, in_host, in_b, cudaMemcpyHostToDevice, c->stream));
  mag_status st = mag_decode_step(c, B, sids, c->d_in_stage, c->d_out_stage);
  if (st != MAG_OK) return st;
  CUDA_TRY(c, cudaMemcpyAsync(out_host, c->d_out_stage, out_b, cudaMemcpyDeviceToHost, c->stream));
  CUDA_TRY(c, cudaStreamSynchronize(c->stream));
  return check_err(c);
}

void mag_adapt_defaults(mag_adapt_config* a) {
  if (!a) return;
  *a = mag_adapt_config{};
  a->enable_adaptive = 1;
  a->adaptive_window_size = 64;
  a->adaptive_sample_rate = 4;
  a->plan_short_below = 128;
  a->plan_long_above = 512;
  // measured on GB300 (8B shape, one session): 4 splits are fastest below ~128 keys, 8 to ~300, 16 above
  a->plan_splits[0] = 4;
  a->plan_splits[1] = 8;
  a->plan_splits[2] = 16;
  a->force_plan = -1;
  a->async_switch = 0;
  a->hot_pool_slack = 1.2f;
}

mag_status mag_set_adaptive(mag_ctx* c, const mag_adapt_config* a) {
  if (!c || !a) return MAG_ERR_INVALID_ARG;
  if (a->enable_adaptive) {
    if (a->adaptive_window_size < 1 || a->adaptive_sample_rate < 1)
      return fail(c, MAG_ERR_INVALID_ARG, "set_adaptive: window %d and sample rate %d must be >= 1",
                  a->adaptive_window_size, a->adaptive_sample_rate);
    if (a->plan_short_below > a->plan_long_above + 1)
      return fail(c, MAG_ERR_INVALID_ARG, "set_adaptive: short_below %d above long_above %d",
                  a->plan_short_below, a->plan_long_above);
    for (int i = 0; i < 3; ++i) {
      if (a->plan_splits[i] < 0 || a->plan_splits[i] > 8 * kAttnMaxGroups)
        return fail(c, MAG_ERR_INVALID_ARG, "set_adaptive: plan %d splits %d not in 0..%d", i, a->plan_splits[i],
                    8 * kAttnMaxGroups);
      if (a->plan_wide[i] != 0 && a->plan_wide[i] != 1)
        return fail(c, MAG_ERR_INVALID_ARG, "set_adaptive: plan %d wide %d not 0 or 1", i, a->plan_wide[i]);
    }
    if (a->force_plan < -1 || a->force_plan > 2)
      return fail(c, MAG_ERR_INVALID_ARG, "set_adaptive: force_plan %d not in -1..2", a->force_plan);
    if (!(a->hot_pool_slack >= 1.0f && a->hot_pool_slack <= 16.0f))
      return fail(c, MAG_ERR_INVALID_ARG, "set_adaptive: hot_pool_slack %g not in 1..16", a->hot_pool_slack);
  }
  mag_status st = finish_capture(c);
  if (st != MAG_OK) return st;
  if (a->enable_adaptive && a->async_switch && !c->cap_stream)
    CUDA_TRY(c, cudaStreamCreateWithFlags(&c->cap_stream, cudaStreamNonBlocking));
  // graphs captured under other split counts are dropped; the ones that stay valid are kept
  mag_adapt_config next = a->enable_adaptive ? *a : mag_adapt_config{};
  for (int p = 0; p < 3; ++p) {
    for (int b = 1; b <= MAG_MAX_BATCH; ++b) {
      const int s_old = plan_splits(c, p, b) * 2 + plan_wide(c, p);
      std::swap(c->adapt, next);
      const int s_new = plan_splits(c, p, b) * 2 + plan_wide(c, p);
      std::swap(c->adapt, next);
      if (s_old == s_new) continue;
      for (int v = 0; v < 2; ++v) {
        mag_ctx::StepGraph& g = c->graphs[v][p][b];
        if (g.exec) {
          CUDA_TRY(c, cudaStreamSynchronize(c->stream));
          CUDA_TRY(c, cudaGraphExecDestroy(g.exec));
          g = mag_ctx::StepGraph{};
        }
      }
    }
  }
  c->adapt = next;
  c->profile.reset();
  if (next.enable_adaptive)
    c->profile = std::make_unique<LoadProfile>(next.adaptive_window_size, next.adaptive_sample_rate);
  c->hot_blocks = -1;
  if (next.enable_adaptive && next.force_plan >= 0) {
    if (next.force_plan != c->cur_plan) ++c->switches;
    c->cur_plan = next.force_plan;
  }
  if (!next.enable_adaptive) c->cur_plan = 1;
  return MAG_OK;
}

mag_status mag_get_profile(mag_ctx* c, mag_profile* out) {
  if (!c || !out) return MAG_ERR_INVALID_ARG;
  mag_status st = poll_capture(c);
  if (st != MAG_OK) return st;
  *out = mag_profile{};
  out->seen = c->profile ? c->profile->seen() : 0;
  out->recorded = c->profile ? c->profile->count() : 0;
  out->p50 = c->profile ? c->profile->quantile(0.5) : -1;
  out->p90 = c->profile ? c->profile->quantile(0.9) : -1;
  out->p99 = c->profile ? c->profile->quantile(0.99) : -1;
  out->plan = c->cur_plan;
  out->pending_plan = c->pending_plan;
  out->plan_splits = plan_splits(c, c->cur_plan, 1);
  out->plan_wide = plan_wide(c, c->cur_plan);
  out->switches = c->switches;
  out->hot_blocks = c->hot_blocks;
  return MAG_OK;
}

}  // extern "C"
