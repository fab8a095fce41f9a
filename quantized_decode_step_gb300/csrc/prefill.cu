// Chunked prefill: set-up of its buffers and activation maps, and the chunk path (one or several sessions).
#include "engine.h"

namespace mag {

// ---------------------------------------------------------------- chunked prefill set-up
// GEMM rows of projection kind i: the tile rows of its 16-row decode tiles, 8 tiles to a 128-row GEMM tile (QKV:
// one head of d = 128 or two of 64, RoPE pairs (i, i + d/2) in canonical order; gate-up: gate and up rows
// interleaved in blocks of 64), padded to a whole GEMM tile.
int prefill_rows(const mag_ctx* c, int i) {
  const int t = tc_gemm_rows_multiple();
  if (i == 2) return (c->F + 63) / 64 * 128;
  const int n = i == 0 ? c->R : c->D;
  return (n + t - 1) / t * t;
}

// Prefill activation tensors at max_chunk rows with their op lifetimes: 0 input, per layer 1 norm,
// 2 QKV, 3 KV store + attention, 4 O, 5 norm, 6 gate-up, 7 down (one plan for every layer); 8 LM head.
void build_prefill_plan(mag_ctx* c) {
  const uint64_t T = c->cfg.max_chunk;
  auto Tn = [](const char* n, uint64_t sz, int f, int l) { return ArenaTensor{n, sz, f, l, 0}; };
  c->pf_plan.clear();
  c->pf_plan.push_back(Tn("pf_residual", T * c->D * 4, 0, 8));
  c->pf_plan.push_back(Tn("pf_norm", T * c->D * 2, 1, 6));
  c->pf_plan.push_back(Tn("pf_qkv", T * c->R * 2, 2, 3));
  c->pf_plan.push_back(Tn("pf_attn_out", T * c->Hq * c->d * 2, 3, 4));
  c->pf_plan.push_back(Tn("pf_ffn_act", T * c->F * 2, 6, 7));
  c->pf_arena_bytes = plan_arena(c->pf_plan, 64, (c->cfg.flags & MAG_FLAG_ARENA_NO_REUSE) != 0);
}

mag_status setup_prefill(mag_ctx* c) {
  cudaError_t e;
  build_prefill_plan(c);
  if ((e = dev_malloc(&c->pf_arena, std::max<uint64_t>(c->pf_arena_bytes, 256))) != cudaSuccess)
    return fail(c, MAG_ERR_OOM, "prefill arena: %s", cudaGetErrorString(e));
  auto at = [&](const char* n) -> uint8_t* {
    for (auto& t : c->pf_plan)
      if (t.name == n) return c->pf_arena + t.offset;
    return nullptr;
  };
  c->pf_r = reinterpret_cast<float*>(at("pf_residual"));
  c->pf_xn = reinterpret_cast<__half*>(at("pf_norm"));
  c->pf_qkv = reinterpret_cast<__half*>(at("pf_qkv"));
  c->pf_o = reinterpret_cast<__half*>(at("pf_attn_out"));
  c->pf_act = reinterpret_cast<__half*>(at("pf_ffn_act"));
  const int T = c->cfg.max_chunk;
  if (!make_tmap_2d(c->map_xn, c->pf_xn, T, c->D) || !make_tmap_2d(c->map_o, c->pf_o, T, (int64_t)c->Hq * c->d) ||
      !make_tmap_2d(c->map_act, c->pf_act, T, c->F))
    return fail(c, MAG_ERR_CUDA, "prefill: activation tensor maps");
  // several sessions in one chunk: per-row positions and sessions, and the gathered last rows
  if ((e = dev_malloc(&c->pf_rows, (size_t)2 * T * 4)) != cudaSuccess ||
      (e = dev_malloc(&c->pf_last_r, (size_t)MAG_MAX_BATCH * c->D * 4)) != cudaSuccess)
    return fail(c, MAG_ERR_OOM, "prefill row tables: %s", cudaGetErrorString(e));
  c->other_bytes += (size_t)2 * T * 4 + (size_t)MAG_MAX_BATCH * c->D * 4;
  // GEMMs whose output blocks fill at most half the SMs split K in two, merged through a workspace
  const size_t pf = tc_gemm_part_floats(c->n_sm), pc = (size_t)(c->n_sm / 2) * 4;
  if ((e = dev_malloc(&c->pf_part, pf * 4)) != cudaSuccess || (e = dev_malloc(&c->pf_part_cnt, pc * 4)) != cudaSuccess)
    return fail(c, MAG_ERR_OOM, "prefill split-K workspace: %s", cudaGetErrorString(e));
  cudaMemsetAsync(c->pf_part_cnt, 0, pc * 4, c->stream);
  c->other_bytes += pf * 4 + pc * 4;
  return MAG_OK;
}

// The chunk path of mag_prefill_chunk and mag_verify_tokens: T tokens of one session through every layer
// (their k and v appended to the pool), then the final RMSNorm + LM head (or the final hidden state) of the
// last out_rows tokens into out [out_rows][V or D].
// One prefill chunk of n_seg sessions: session sids[i] appends ntok[i] tokens, the rows of the sessions
// following each other in `in` ([sum ntok][D]); each session's tokens attend causally to its own cache.
// Output: with all_rows (one session), every row; otherwise the last row of every session, in order.
// With resid_dump (debug) the launches run without programmatic dependent launch and the fp32 residual of
// the T rows is copied there after the input and after every layer: [L+1][T][D].
mag_status run_chunk(mag_ctx* c, const char* what, int n_seg, const int32_t* sids, const int32_t* ntok,
                     const void* in, void* out, bool all_rows, float* resid_dump) {
  if (!c) return MAG_ERR_INVALID_ARG;
  if (c->cfg.max_chunk <= 0) return fail(c, MAG_ERR_UNSUPPORTED, "%s: created with max_chunk = 0", what);
  if (!in || !out || !sids || !ntok) return fail(c, MAG_ERR_INVALID_ARG, "%s: null buffer", what);
  if (n_seg < 1 || n_seg > MAG_MAX_BATCH)
    return fail(c, MAG_ERR_INVALID_ARG, "%s: %d sessions not in 1..%d", what, n_seg, MAG_MAX_BATCH);
  if (!all_loaded(c)) return fail(c, MAG_ERR_NOT_LOADED, "%s: not every weight is loaded", what);
  int T = 0, need = 0;
  for (int i = 0; i < n_seg; ++i) {
    const int sid = sids[i];
    if (sid < 0 || sid >= (int)c->sessions.size() || !c->sessions[sid].open)
      return fail(c, MAG_ERR_INVALID_ARG, "%s: session %d is not open", what, sid);
    for (int j = 0; j < i; ++j)
      if (sids[j] == sid) return fail(c, MAG_ERR_INVALID_ARG, "%s: session %d appears twice", what, sid);
    if (ntok[i] < 1 || ntok[i] > c->cfg.max_chunk - T)
      return fail(c, MAG_ERR_INVALID_ARG, "%s: %d + %d tokens exceed max_chunk %d", what, T, ntok[i],
                  c->cfg.max_chunk);
    const Session& s = c->sessions[sid];
    if ((int64_t)s.len + ntok[i] > c->cfg.max_context)
      return fail(c, MAG_ERR_CONTEXT_FULL, "%s: %d + %d tokens exceed max_context %d", what, s.len, ntok[i],
                  c->cfg.max_context);
    T += ntok[i];
    need += (s.len + ntok[i] + 15) / 16 - (s.len + 15) / 16;
  }
  const int out_rows = all_rows ? T : n_seg;
  if (all_rows && (n_seg != 1 || T > kPipeMaxBatch))
    return fail(c, MAG_ERR_INVALID_ARG, "%s: every row's output needs one session of 1..%d tokens", what,
                kPipeMaxBatch);
  mag_status rs = reserve_blocks(c, what, need);
  if (rs != MAG_OK) return rs;
  {
    int32_t keys[MAG_MAX_BATCH];
    for (int i = 0; i < n_seg; ++i) keys[i] = c->sessions[sids[i]].len + ntok[i];
    rs = stats_begin(c, 2, T, out_rows, keys, n_seg);
    if (rs != MAG_OK) return rs;
  }
  // step arguments of the output rows' LM head (or final hidden state)
  const int slot = c->ring_pos;
  CUDA_TRY(c, cudaEventSynchronize(c->ring_ev[slot]));
  StepArgs& sa = c->h_ring[slot];
  memset(&sa, 0, sizeof sa);
  sa.batch = out_rows;
  sa.out = out;
  PrefillAttnArgs pa = {};
  pa.err = c->d_err;
  pa.n_seg = n_seg;
  RowList last = {};
  last.n = n_seg;
  std::vector<int32_t> rows;  // [2][T]: position and session of every row, several sessions only
  if (n_seg > 1) rows.resize((size_t)2 * T);
  for (int i = 0, row0 = 0; i < n_seg; row0 += ntok[i], ++i) {
    Session& s = c->sessions[sids[i]];
    pa.seg[i] = PfSeg{row0, ntok[i], s.len, sids[i]};
    last.row[i] = row0 + ntok[i] - 1;
    if (n_seg > 1)
      for (int t = 0; t < ntok[i]; ++t) {
        rows[row0 + t] = s.len + t;
        rows[(size_t)T + row0 + t] = sids[i];
      }
    const int nb_old = (s.len + 15) / 16, nb_new = (s.len + ntok[i] + 15) / 16;
    for (int b = nb_old; b < nb_new; ++b) s.table.push_back(c->kv.pop());
    int32_t* row = c->d_tables + (size_t)sids[i] * c->table_stride;
    if (nb_new > nb_old)
      CUDA_TRY(c, cudaMemcpyAsync(row + nb_old, s.table.data() + nb_old, (size_t)(nb_new - nb_old) * 4,
                                  cudaMemcpyHostToDevice, c->stream));
  }
  for (int b = 0; b < out_rows; ++b) {
    sa.sess[b] = all_rows ? sids[0] : sids[b];
    sa.pos[b] = all_rows ? c->sessions[sids[0]].len + b : c->sessions[sids[b]].len + ntok[b] - 1;
  }
  if (n_seg > 1)  // pageable source: the copy has taken the bytes when the call returns
    CUDA_TRY(c, cudaMemcpyAsync(c->pf_rows, rows.data(), rows.size() * 4, cudaMemcpyHostToDevice, c->stream));
  CUDA_TRY(c, cudaMemcpyAsync(c->d_args, &sa, sizeof sa, cudaMemcpyHostToDevice, c->stream));
  CUDA_TRY(c, cudaEventRecord(c->ring_ev[slot], c->stream));
  c->ring_pos = (slot + 1) % kRing;
  const int32_t* row_pos = n_seg > 1 ? c->pf_rows : nullptr;
  const int32_t* row_sess = n_seg > 1 ? c->pf_rows + T : nullptr;
  const int p0 = c->sessions[sids[0]].len;  // one session: positions p0 + row
  int32_t* row = c->d_tables + (size_t)sids[0] * c->table_stride;

  int n = 0;
  const bool pdl = !(c->cfg.flags & MAG_FLAG_NO_PDL) && !resid_dump;
  Launch L{c->stream, pdl, &n};
  const int D = c->D, HD = c->Hq * c->d;
  const PoolGeom pg = pool_geom(c);
  auto dump = [&](int i) {
    return resid_dump ? cudaMemcpyAsync(resid_dump + (size_t)i * T * D, c->pf_r, (size_t)T * D * 4,
                                        cudaMemcpyDeviceToDevice, c->stream)
                      : cudaSuccess;
  };
  CUDA_TRY(c, launch_rows_to_resid(L, (const __half*)in, c->pf_r, T, D));
  CUDA_TRY(c, dump(0));
  for (int l = 0; l < c->L; ++l) {
    const Proj* P = &c->proj[(size_t)l * 4];
    TcGemmArgs g = {};
    g.M = T;
    g.err = c->d_err;
    g.wait_limit = c->wait_limit;
    // the GEMM's weights: projection i's decode tiles, their rows in the order its epilogue wants
    auto weights = [&](TcGemmArgs& x, int i) {
      const Proj& pr = P[i];
      x.w = pr.tiles;
      x.n_dtiles = pr.N / 16;
      x.C = (pr.K + 63) / 64;
      x.N = prefill_rows(c, i);
      x.K = pr.K;
      x.ksplit = tc_gemm_ksplit(x.M, x.N, x.K, c->n_sm);
      x.part = c->pf_part;
      x.part_cnt = c->pf_part_cnt;
      if (pr.map == MAP_QKV) {
        x.tpg = c->d / 16, x.gsz = c->d, x.half = c->d / 2;
      } else if (pr.map == MAP_SWIGLU) {
        x.tpg = 8, x.gsz = 128, x.half = 64;
      } else {
        x.tpg = 1, x.gsz = 16, x.half = 8;
      }
    };
    // RMSNorm + QKV (+ RoPE of q and k)
    CUDA_TRY(c, launch_rmsnorm_rows(L, c->pf_r, c->gamma1[l], c->cfg.rms_eps, T, D, c->pf_xn));
    TcGemmArgs gq = g;
    weights(gq, 0);
    gq.n_valid = c->R;
    gq.out = c->pf_qkv;
    gq.ldo = c->R;
    gq.head_dim = c->d;
    gq.n_rot_heads = c->Hq + c->Hkv;
    gq.pos0 = p0;
    gq.row_pos = row_pos;
    gq.rope_cos = c->d_cos;
    gq.rope_sin = c->d_sin;
    CUDA_TRY(c, launch_tc_gemm(L, c->map_xn, gq, EPI_QKV));
    // the chunk's k, v into the pool, then causal attention over the pool
    KvChunkArgs kc = {};
    kc.err = c->d_err;
    kc.qkv = c->pf_qkv;
    kc.qkv_ld = c->R;
    kc.n_heads = c->Hq;
    kc.n_tok = T;
    kc.pos0 = p0;
    kc.layer = l;
    kc.table = row;
    kc.pool = pg;
    kc.row_pos = row_pos;
    kc.row_sess = row_sess;
    CUDA_TRY(c, launch_kv_store_chunk(L, kc));
    pa.qkv = c->pf_qkv;
    pa.qkv_ld = c->R;
    pa.o = c->pf_o;
    pa.ldo = HD;
    pa.n_heads = c->Hq;
    pa.n_kv_heads = c->Hkv;
    pa.head_dim = c->d;
    pa.layer = l;
    pa.pool = pg;
    CUDA_TRY(c, launch_prefill_attention(L, pa));
    // O projection + residual
    TcGemmArgs go = g;
    weights(go, 1);
    go.n_valid = D;
    go.r = c->pf_r;
    go.ldr = D;
    CUDA_TRY(c, launch_tc_gemm(L, c->map_o, go, EPI_RESID));
    // RMSNorm + gate-up + SwiGLU
    CUDA_TRY(c, launch_rmsnorm_rows(L, c->pf_r, c->gamma2[l], c->cfg.rms_eps, T, D, c->pf_xn));
    TcGemmArgs gg = g;
    weights(gg, 2);
    gg.n_valid = c->F;
    gg.out = c->pf_act;
    gg.ldo = c->F;
    CUDA_TRY(c, launch_tc_gemm(L, c->map_xn, gg, EPI_SWIGLU));
    // down projection + residual
    TcGemmArgs gd = g;
    weights(gd, 3);
    gd.n_valid = D;
    gd.r = c->pf_r;
    gd.ldr = D;
    CUDA_TRY(c, launch_tc_gemm(L, c->map_act, gd, EPI_RESID));
    CUDA_TRY(c, dump(l + 1));
  }
  // the output rows: contiguous for one session, else each session's last row gathered
  float* r_out = c->pf_r + (size_t)(T - out_rows) * D;
  if (n_seg > 1) {
    CUDA_TRY(c, launch_gather_rows(L, c->pf_r, D, last, c->pf_last_r));
    r_out = c->pf_last_r;
  }
  if (c->V) {  // final RMSNorm + LM head of the output rows
    GemvArgs a = gemv_args(c, 4, reinterpret_cast<const uint8_t*>(c->lm_head), c->V / 16, D, out_rows);
    a.r = r_out;
    a.ldr = D;
    a.gamma = c->gamma_f;
    a.ldo = c->V;
    CUDA_TRY(c, launch_gemv(L, a, W_F16, XSRC_RESID, EPI_STORE_OUT));
  } else {
    CUDA_TRY(c, launch_final_hidden(L, c->d_args, r_out, D, out_rows));
  }
  c->last_launches = n;
  for (int i = 0; i < n_seg; ++i) c->sessions[sids[i]].len += ntok[i];
  return stats_end(c);
}

}  // namespace mag

extern "C" {

mag_status mag_prefill_chunk(mag_ctx* c, int32_t sid, int32_t T, const void* in, void* last_out) {
  return run_chunk(c, "prefill_chunk", 1, &sid, &T, in, last_out, false);
}

mag_status mag_debug_prefill_residuals(mag_ctx* c, int32_t sid, int32_t T, const void* in, void* last_out,
                                       void* resid) {
  if (!c) return MAG_ERR_INVALID_ARG;
  if (!resid) return fail(c, MAG_ERR_INVALID_ARG, "debug_prefill_residuals: null residual buffer");
  mag_status st = run_chunk(c, "debug_prefill_residuals", 1, &sid, &T, in, last_out, false,
                            static_cast<float*>(resid));
  if (st != MAG_OK) return st;
  CUDA_TRY(c, cudaStreamSynchronize(c->stream));
  return check_err(c);
}

mag_status mag_prefill_batch(mag_ctx* c, int32_t n_sessions, const int32_t* sids, const int32_t* n_tokens,
                             const void* in, void* last_out) {
  return run_chunk(c, "prefill_batch", n_sessions, sids, n_tokens, in, last_out, false);
}

}  // extern "C"
