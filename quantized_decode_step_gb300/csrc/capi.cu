// C ABI of the decode-step library: context, weights, KV block pool, sessions, statistics and the debug
// hooks (the decode step: step.cu; chunked prefill: prefill.cu; the verify step: verify.cu). See
// include/mag.h for the contract of each call.
#include "engine.h"

namespace mag {

mag_status fail(mag_ctx* c, mag_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (c) c->err = buf;
  return s;
}

// After a synchronisation: a kernel whose bounded wait gave up left a bit in the error word.
// The arrival counters of the last-to-arrive merges (GEMV tiles, attention clusters, prefill split-K) may be
// left part-way by a role that gave up: they start again from zero.
mag_status check_err(mag_ctx* c) {
  const uint32_t e = *reinterpret_cast<volatile uint32_t*>(c->h_err);
  if (e == 0) return MAG_OK;
  *reinterpret_cast<volatile uint32_t*>(c->h_err) = 0;
  if (e & (kErrCanary | kErrBounds)) {
    std::string what;
    if (e & kErrCanary) {
      what = "a canary band changed around arena tensor(s):";
      for (size_t i = 0; i < c->plan.size() && i < 16; ++i)
        if (e & (1u << (kErrCanaryShift + i))) what += " " + c->plan[i].name;
      // the bands again, for the steps after this one
      for (const auto& t : c->plan) {
        cudaMemsetAsync(c->arena + t.offset, kCanaryByte, c->canary_band, c->stream);
        cudaMemsetAsync(c->arena + t.offset + t.size - c->canary_band, kCanaryByte, c->canary_band, c->stream);
      }
    }
    if (e & kErrBounds) {
      if (!what.empty()) what += "; ";
      what += "a block-table entry outside the pool (not used; the step's results are wrong)";
      // the device tables from the host's copy
      for (size_t sid = 0; sid < c->sessions.size(); ++sid)
        if (c->sessions[sid].open && !c->sessions[sid].table.empty())
          cudaMemcpyAsync(c->d_tables + sid * c->table_stride, c->sessions[sid].table.data(),
                          c->sessions[sid].table.size() * 4, cudaMemcpyHostToDevice, c->stream);
    }
    cudaStreamSynchronize(c->stream);
    return fail(c, MAG_ERR_CORRUPT, "%s", what.c_str());
  }
  cudaMemsetAsync(c->d_counters, 0, c->n_counters * 4, c->stream);
  cudaMemsetAsync(c->attn_arrivals, 0, (size_t)c->B_max * c->Hkv * 4, c->stream);
  if (c->pf_part_cnt) cudaMemsetAsync(c->pf_part_cnt, 0, (size_t)(c->n_sm / 2) * 4 * 4, c->stream);
  return fail(c, MAG_ERR_TIMEOUT, "a kernel's pipeline wait gave up (code 0x%x)", e);
}

// Launch shape of one projection at batch B. Up to kPipeMaxBatch tokens: the
// pipelined kernel, one block per SM over contiguous tile ranges, its per-warp
// rings as deep as a shared-memory budget allows. W4 above that: k-windows whose
// staged activations fit in 64 KB, times tile ranges, about one block per SM,
// rings as deep as the rest of the block's shared memory allows. The fp16 LM
// head above 4 tokens: a k-split grid of 8-warp blocks.

GemvPlan plan_gemv(const mag_ctx* c, int kind, int n_mtiles, int K, int B) {
  GemvPlan p = {};
  const int n_chunks = (K + 63) / 64;
  if (B <= kPipeMaxBatch) {
    const int wfmt = kind == 4 ? W_F16 : W_W4;
    p.n_cta = std::max(1, std::min(c->n_sm, n_mtiles));
    p.t_max = (n_mtiles + p.n_cta - 1) / p.n_cta;
    const size_t base = gemv_pipe_smem_bytes(wfmt, B, n_chunks, 0, p.t_max);
    const size_t stage = gemv_pipe_slot_bytes(wfmt);
    const size_t budget = kPipeBudget;
    const int fit = budget > base ? (int)((budget - base) / stage) : 0;
    p.stages = std::max(2, std::min(gemv_pipe_max_stages(), fit));
    p.smem = gemv_pipe_smem_bytes(wfmt, B, n_chunks, p.stages, p.t_max);
    p.ks = 1;
    p.cpc = n_chunks;
    return p;
  }
  if (kind != 4) {
    // window: a multiple of 4 chunks whose B token rows fit in 64 KB of fp16
    const int cw_max = std::max(4, (int)((64 * 1024) / ((size_t)B * 128)) / 4 * 4);
    const int kw0 = (n_chunks + cw_max - 1) / cw_max;
    // windows x tile ranges closest to one block per SM (fewest windows on a tie)
    int best_kw = kw0, best_blocks = 0;
    for (int kw = kw0; kw <= kw0 + 3; ++kw) {
      const int cw = ((n_chunks + kw - 1) / kw + 3) / 4 * 4;
      const int kw_eff = (n_chunks + cw - 1) / cw;
      const int tr = std::max(1, std::min(n_mtiles, c->n_sm / kw_eff));
      if (kw != kw0 && kw_eff * tr > c->n_sm) continue;  // more windows only while they fill idle SMs
      if (kw_eff * tr > best_blocks) {
        best_blocks = kw_eff * tr;
        best_kw = kw_eff;
      }
    }
    p.cpc = ((n_chunks + best_kw - 1) / best_kw + 3) / 4 * 4;
    p.ks = (n_chunks + p.cpc - 1) / p.cpc;
    p.n_cta = std::max(1, std::min(n_mtiles, c->n_sm / p.ks));
    p.t_max = (n_mtiles + p.n_cta - 1) / p.n_cta;
    const size_t base = gemv_batch_smem_bytes(B, p.cpc, 0, p.t_max);
    const size_t stage = gemv_batch_stage_bytes();
    const int fit = kSmemMax > base ? (int)((kSmemMax - base) / stage) : 0;
    p.stages = std::max(2, std::min(gemv_batch_max_stages(), fit));
    p.smem = gemv_batch_smem_bytes(B, p.cpc, p.stages, p.t_max);
    return p;
  }
  const int max_cpc = std::max(1, (64 * 1024) / (B * 136) - 1);
  p.ks = (n_chunks + max_cpc - 1) / max_cpc;
  p.cpc = (n_chunks + p.ks - 1) / p.ks;
  // tiles per warp: the fewest that keep the grid within one wave of two blocks per SM (each block
  // stages its k-range of activations once for all its tiles)
  const int groups = (n_mtiles + 7) / 8;
  p.tpw = 1;
  while (p.tpw < 4 && (int64_t)((groups + p.tpw - 1) / p.tpw) * p.ks > 2 * c->n_sm) p.tpw *= 2;
  return p;
}

// Splits of one (session, KV head): the blocks of one thread-block cluster, so at
// most the largest cluster the device co-schedules (16 on a full GPU).
int attn_splits(const mag_ctx* c, int B, bool wide) {
  int s = (2 * c->n_sm + B * c->Hkv - 1) / (B * c->Hkv);
  return std::max(1, std::min(s, wide ? c->attn_cluster_max_wide : c->attn_cluster_max));
}

int64_t kv_data_bytes(int d, int dt) { return dt == 0 ? 2 * d : (dt == 1 ? d : d / 2); }
int64_t kv_meta_bytes(int d, int dt) { return dt == 0 ? 0 : (dt == 1 ? 2 : (d / 32) * 4); }

PoolGeom pool_geom(const mag_ctx* c) {
  PoolGeom g;
  g.base = c->kv.base();
  g.block_bytes = c->block_bytes;
  g.pool_blocks = c->cfg.pool_blocks;
  g.data_bytes = c->data_bytes;
  g.meta_bytes = c->meta_bytes;
  g.n_kv_heads = c->Hkv;
  g.head_dim = c->d;
  g.kv_dtype = c->cfg.kv_dtype;
  g.tables = c->d_tables;
  g.table_stride = c->table_stride;
  return g;
}

// Make n pool blocks free and mapped; an error leaves the context unchanged.
mag_status reserve_blocks(mag_ctx* c, const char* what, int64_t n) {
  const mag_status st = c->kv.reserve(n, c->stream);
  if (st == MAG_ERR_KV_FULL)
    return fail(c, st, "%s: needs %lld blocks, %lld free", what, (long long)n, (long long)c->kv.available());
  if (st != MAG_OK) return fail(c, st, "%s: %s", what, c->kv.err.c_str());
  return MAG_OK;
}

// Whether an open session lists a block of group g of an elastic pool (checked before the group's release).
bool group_referenced(const mag_ctx* c, int64_t g) {
  const int64_t G = c->kv.group_blocks();
  for (const Session& s : c->sessions)
    if (s.open)
      for (int32_t b : s.table)
        if (b / G == g) return true;
  return false;
}

// Elastic pool: release free groups above the hot size, unmap released ones the stream has passed.
mag_status pool_trim(mag_ctx* c) {
  if (!c->kv.elastic()) return MAG_OK;
  const mag_status st = c->kv.trim(c->stream, [c](int64_t g) { return group_referenced(c, g); });
  return st == MAG_OK ? st : fail(c, st, "%s", c->kv.err.c_str());
}

bool all_loaded(const mag_ctx* c) {
  for (int l = 0; l < c->L; ++l)
    for (int i = 0; i < 6; ++i)
      if (!c->loaded[l * 6 + i]) return false;
  if (!c->loaded[c->L * 6]) return false;
  if (c->V && !c->loaded[c->L * 6 + 1]) return false;
  return true;
}

std::vector<ProjShape> proj_shapes(const mag_ctx* c) {
  std::vector<ProjShape> v = {{0, c->R / 16, c->D, W_W4, XSRC_RESID, EPI_QKV},
                              {1, c->D / 16, c->Hq * c->d, W_W4, XSRC_F16, EPI_RESID},
                              {2, c->F / 8, c->D, W_W4, XSRC_RESID, EPI_SWIGLU},
                              {3, c->D / 16, c->F, W_W4, XSRC_F16, EPI_RESID}};
  if (c->V) v.push_back({4, c->V / 16, c->D, W_F16, XSRC_RESID, EPI_STORE_OUT});
  return v;
}

// Floats of the partial-sum buffer for batch B (k-split slices).
size_t gemv_partial_floats(const mag_ctx* c, int B) {
  size_t mx = 0;
  const int nt = B > 8 ? 2 : 1;
  for (auto& ps : proj_shapes(c)) {
    GemvPlan p = plan_gemv(c, ps.kind, ps.n_mtiles, ps.K, B);
    if (B > kPipeMaxBatch && p.ks > 1) mx = std::max(mx, (size_t)p.ks * ps.n_mtiles * 32 * 4 * nt);
  }
  return mx;
}

// Shared memory of the pipelined kernel for every projection and batch must fit one block.
bool gemv_plans_fit(const mag_ctx* c, std::string& why) {
  for (auto& ps : proj_shapes(c))
    for (int B = 1; B <= c->B_max; ++B) {
      const GemvPlan p = plan_gemv(c, ps.kind, ps.n_mtiles, ps.K, B);
      if (p.smem > kSmemMax) {
        char b[160];
        snprintf(b, sizeof b, "projection %d (K = %d) at batch %d needs %zu bytes of shared memory (limit %zu)",
                 ps.kind, ps.K, B, p.smem, kSmemMax);
        why = b;
        return false;
      }
    }
  return true;
}

// Counter slots: one per tile (W4 k-windows) or block column (fp16 k-split).
size_t gemv_counters(const mag_ctx* c) {
  size_t mx = 1;
  for (auto& ps : proj_shapes(c)) mx = std::max(mx, (size_t)ps.n_mtiles);
  return mx;
}

// Decode-phase activation tensors at max_batch with their op lifetimes: op 0
// step begin; per layer 1 QKV, 2 attention, 3 O, 4 gate-up, 5 down (one plan,
// reused by every layer); 6 LM head.
void build_decode_plan(mag_ctx* c) {
  const int B = c->B_max;
  size_t part = 0;
  for (int b = 1; b <= B; ++b) part = std::max(part, gemv_partial_floats(c, b));
  auto T = [](const char* n, uint64_t sz, int f, int l) { return ArenaTensor{n, sz, f, l, 0}; };
  c->plan.clear();
  c->plan.push_back(T("residual", (uint64_t)B * c->D * 4, 0, 6));
  c->plan.push_back(T("sumsq_part", (uint64_t)(c->D / 16) * MAG_MAX_BATCH * 4, 0, 6));
  c->plan.push_back(T("qkv", (uint64_t)B * c->R * 2, 1, 2));
  c->plan.push_back(T("attn_out", (uint64_t)B * c->Hq * c->d * 2, 2, 3));
  c->plan.push_back(T("ffn_act", (uint64_t)B * c->F * 2, 4, 5));
  if (part) c->plan.push_back(T("gemv_partial", part * 4, 1, 6));
  c->arena_unshared = 0;
  for (auto& t : c->plan) c->arena_unshared += t.size;
  // debug canaries: every tensor between two bands of its own, and no two tensors share bytes (a tensor's
  // bytes may then not be another one's band)
  const bool canary = (c->cfg.flags & MAG_FLAG_DEBUG_CANARY) != 0;
  c->canary_band = canary ? kCanaryBand : 0;
  for (auto& t : c->plan) t.size += 2 * c->canary_band;
  c->arena_bytes = plan_arena(c->plan, 64, canary || (c->cfg.flags & MAG_FLAG_ARENA_NO_REUSE) != 0);
}

void* arena_ptr(mag_ctx* c, const char* name) {
  for (auto& t : c->plan)
    if (t.name == name) return c->arena + t.offset + c->canary_band;
  return nullptr;
}

ArenaCheck arena_check_args(const mag_ctx* c) {
  ArenaCheck a = {};
  a.base = c->arena;
  a.err = c->d_err;
  for (const auto& t : c->plan) {
    if (a.n == 16) break;
    a.band[a.n][0] = t.offset;
    a.band[a.n][1] = t.offset + t.size - c->canary_band;
    ++a.n;
  }
  return a;
}

GemvArgs gemv_args(const mag_ctx* c, int kind, const uint8_t* w, int n_mtiles, int K, int B) {
  GemvArgs a = {};
  GemvPlan pl = plan_gemv(c, kind, n_mtiles, K, B);
  a.w = w;
  a.n_mtiles = n_mtiles;
  a.K = K;
  a.n_chunks = (K + 63) / 64;
  a.n_cta = pl.n_cta;
  a.stages = pl.stages;
  a.t_max = pl.t_max;
  a.err = c->d_err;
  a.wait_limit = c->wait_limit;
  a.chunks_per_cta = pl.cpc;
  a.ks = pl.ks;
  a.tpw = pl.tpw;
  a.batch = B;
  a.eps = c->cfg.rms_eps;
  a.r = c->r;
  a.ldr = c->D;
  a.ss_part = c->ss_part;
  a.n_ss = c->D / 16;
  a.partial = c->gemv_part;
  a.counters = c->d_counters;
  a.step = c->d_args;
  a.trace = c->trace;
  return a;
}

void free_ctx(mag_ctx* c) {
  if (!c) return;
  if (c->stream) cudaStreamSynchronize(c->stream);
  if (c->cap_thread.joinable()) c->cap_thread.join();
  for (auto& gv : c->graphs)
    for (auto& gp : gv)
      for (auto& g : gp)
        if (g.exec) cudaGraphExecDestroy(g.exec);
  for (auto& gv : c->len_graphs)
    for (auto& gp : gv)
      for (auto& g : gp)
        if (g.exec) cudaGraphExecDestroy(g.exec);
  if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
  for (auto& e : c->ring_ev)
    if (e) cudaEventDestroy(e);
  for (auto& e : c->ev_step)
    if (e) cudaEventDestroy(e);
  cudaFree(c->wbase);
  cudaFree(c->d_tables);
  cudaFree(c->d_cos);
  cudaFree(c->d_sin);
  cudaFree(c->arena);
  cudaFree(c->d_counters);
  cudaFree(c->trace_n);
  cudaFree(c->attn_part);
  cudaFree(c->attn_arrivals);
  cudaFree(c->d_args);
  cudaFree(c->d_in_stage);
  cudaFree(c->d_out_stage);
  if (c->h_ring) cudaFreeHost(c->h_ring);
  if (c->h_err) cudaFreeHost(c->h_err);
  cudaFree(c->pf_arena);
  cudaFree(c->pf_rows);
  cudaFree(c->pf_part);
  cudaFree(c->pf_part_cnt);
  cudaFree(c->pf_last_r);
  if (c->own_stream && c->stream) cudaStreamDestroy(c->stream);
  delete c;
}

mag_status check_cfg(const mag_config* g, std::string& why) {
  char b[256];
  auto bad = [&](const char* m) {
    why = m;
    return MAG_ERR_INVALID_ARG;
  };
  if (g->n_layers < 1 || g->hidden < 16 || g->n_heads < 1 || g->n_kv_heads < 1 || g->ffn < 8 || g->vocab < 0)
    return bad("shape fields must be positive (vocab >= 0)");
  if (g->n_heads % g->n_kv_heads) return bad("n_heads must be a multiple of n_kv_heads");
  if (g->n_heads / g->n_kv_heads > 8) return bad("more than 8 query heads per KV head");
  if (g->head_dim != 64 && g->head_dim != 128) return bad("head_dim must be 64 or 128");
  if (g->hidden % 16 || g->ffn % 8 || (g->n_heads * g->head_dim) % 16) return bad("hidden % 16, ffn % 8 required");
  if (g->vocab % 16) return bad("vocab must be a multiple of 16");
  if (g->block_tokens != 16) return bad("block_tokens must be 16");
  if (g->kv_dtype < 0 || g->kv_dtype > 2) return bad("kv_dtype must be 0 (FP16), 1 (INT8) or 2 (INT4)");
  if (g->pool_blocks < 1 || g->max_sessions < 1 || g->max_context < 1) return bad("pool, sessions, context > 0");
  if (g->max_batch < 1 || g->max_batch > MAG_MAX_BATCH) return bad("max_batch must be 1..16");
  if (g->max_chunk < 0) return bad("max_chunk must be >= 0");
  if (!(g->rms_eps > 0) || !(g->rope_base > 0)) return bad("rms_eps and rope_base must be positive");
  snprintf(b, sizeof b, "ok");
  return MAG_OK;
}

}  // namespace mag

// ============================================================================ API

extern "C" {

mag_status mag_create(const mag_config* cfg, void* cuda_stream, mag_ctx** out) {
  if (!out) return MAG_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg) return MAG_ERR_INVALID_ARG;
  std::string why;
  if (check_cfg(cfg, why) != MAG_OK) {
    fprintf(stderr, "mag_create: %s\n", why.c_str());
    return MAG_ERR_INVALID_ARG;
  }
  mag_ctx* c = new mag_ctx();
  c->cfg = *cfg;
  c->cfg.pool_order_host = nullptr;
  c->L = cfg->n_layers;
  c->D = cfg->hidden;
  c->Hq = cfg->n_heads;
  c->Hkv = cfg->n_kv_heads;
  c->d = cfg->head_dim;
  c->F = cfg->ffn;
  c->V = cfg->vocab;
  c->G = c->Hq / c->Hkv;
  c->R = (c->Hq + 2 * c->Hkv) * c->d;
  c->B_max = cfg->max_batch;
  c->table_stride = (cfg->max_context + 15) / 16;
  auto bail = [&](mag_status s) {
    fprintf(stderr, "mag_create: %s\n", c->err.c_str());
    free_ctx(c);
    return s;
  };
  cudaError_t e;
  if ((e = cudaGetDevice(&c->device)) != cudaSuccess) {
    fail(c, MAG_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    return bail(MAG_ERR_CUDA);
  }
  cudaDeviceGetAttribute(&c->n_sm, cudaDevAttrMultiProcessorCount, c->device);
  if ((e = attention_max_cluster(cfg->head_dim, cfg->kv_dtype, false, &c->attn_cluster_max)) != cudaSuccess ||
      (e = attention_max_cluster(cfg->head_dim, cfg->kv_dtype, true, &c->attn_cluster_max_wide)) != cudaSuccess) {
    fail(c, MAG_ERR_CUDA, "attention cluster query: %s", cudaGetErrorString(e));
    return bail(MAG_ERR_CUDA);
  }
  if (cuda_stream) {
    c->stream = (cudaStream_t)cuda_stream;
  } else {
    if ((e = cudaStreamCreate(&c->stream)) != cudaSuccess) {
      fail(c, MAG_ERR_CUDA, "cudaStreamCreate: %s", cudaGetErrorString(e));
      return bail(MAG_ERR_CUDA);
    }
    c->own_stream = true;
  }
  // pool order (a fixed pool only: an elastic one hands out the lowest free block)
  const int P = cfg->pool_blocks;
  if (cfg->pool_order_host) {
    if (cfg->flags & MAG_FLAG_ELASTIC_POOL) {
      fail(c, MAG_ERR_INVALID_ARG, "pool_order_host is not used with MAG_FLAG_ELASTIC_POOL");
      return bail(MAG_ERR_INVALID_ARG);
    }
    std::vector<char> seen(P, 0);
    for (int i = 0; i < P; ++i) {
      int b = cfg->pool_order_host[i];
      if (b < 0 || b >= P || seen[b]) {
        fail(c, MAG_ERR_INVALID_ARG, "pool_order_host is not a permutation of 0..%d", P - 1);
        return bail(MAG_ERR_INVALID_ARG);
      }
      seen[b] = 1;
    }
  }
  c->sessions.resize(cfg->max_sessions);
  c->loaded.assign((size_t)c->L * 6 + 2, 0);

  // ---- weights region: W4 projections as 640-byte tiles, fp16 gains, fp16 LM head
  size_t off = 0;
  c->proj.resize((size_t)c->L * 4);
  std::vector<size_t> offs;
  const int shapes[4][2] = {{c->R, c->D}, {c->D, c->Hq * c->d}, {2 * c->F, c->D}, {c->D, c->F}};
  const int maps[4][2] = {{MAP_QKV, c->d}, {MAP_PLAIN, 0}, {MAP_SWIGLU, c->F}, {MAP_PLAIN, 0}};
  for (int l = 0; l < c->L; ++l)
    for (int i = 0; i < 4; ++i) {
      Proj& p = c->proj[(size_t)l * 4 + i];
      p.N = shapes[i][0];
      p.K = shapes[i][1];
      p.G = (p.K + 31) / 32;
      p.map = maps[i][0];
      p.map_arg = maps[i][1];
      p.canon_bytes = (size_t)p.N * p.G * 20;
      p.tile_bytes = (size_t)(p.N / 16) * ((p.K + 63) / 64) * kTileBytes;
      offs.push_back(off);
      off = align256(off + p.tile_bytes);
    }
  std::vector<size_t> goffs;
  for (int l = 0; l < c->L; ++l)
    for (int i = 0; i < 2; ++i) {
      goffs.push_back(off);
      off = align256(off + (size_t)c->D * 2);
    }
  size_t gf_off = off;
  off = align256(off + (size_t)c->D * 2);
  size_t lm_off = off;
  if (c->V) off = align256(off + (size_t)(c->V / 16) * ((c->D + 63) / 64) * 2048);  // fp16 tiles, ragged k zeroed
  c->wbytes = off;
  if ((e = dev_malloc(&c->wbase, c->wbytes)) != cudaSuccess) {
    fail(c, MAG_ERR_OOM, "weights: device allocation of %zu bytes: %s", c->wbytes, cudaGetErrorString(e));
    return bail(MAG_ERR_OOM);
  }
  for (size_t i = 0; i < c->proj.size(); ++i) c->proj[i].tiles = c->wbase + offs[i];
  for (int l = 0; l < c->L; ++l) {
    c->gamma1.push_back(reinterpret_cast<__half*>(c->wbase + goffs[2 * l]));
    c->gamma2.push_back(reinterpret_cast<__half*>(c->wbase + goffs[2 * l + 1]));
  }
  c->gamma_f = reinterpret_cast<__half*>(c->wbase + gf_off);
  c->lm_head = c->V ? reinterpret_cast<__half*>(c->wbase + lm_off) : nullptr;

  // ---- KV pool (zeroed: slots past a session's length read as finite zeros)
  c->data_bytes = (int)kv_data_bytes(c->d, cfg->kv_dtype);
  c->meta_bytes = (int)kv_meta_bytes(c->d, cfg->kv_dtype);
  c->block_bytes = 2 * (int64_t)c->Hkv * 16 * (c->data_bytes + c->meta_bytes);
  {
    const mag_status st = (cfg->flags & MAG_FLAG_ELASTIC_POOL)
                              ? c->kv.init_elastic(c->L, P, c->block_bytes, c->device, c->stream)
                              : c->kv.init_fixed(c->L, P, c->block_bytes, cfg->pool_order_host, c->stream);
    if (st != MAG_OK) {
      fail(c, st, "%s", c->kv.err.c_str());
      return bail(st);
    }
    c->cfg.pool_blocks = (int32_t)c->kv.blocks();  // elastic: rounded up to whole mapping groups
  }
  size_t tb = (size_t)cfg->max_sessions * c->table_stride * 4;
  if ((e = dev_malloc(&c->d_tables, tb)) != cudaSuccess) {
    fail(c, MAG_ERR_OOM, "block tables: %s", cudaGetErrorString(e));
    return bail(MAG_ERR_OOM);
  }
  cudaMemsetAsync(c->d_tables, 0, tb, c->stream);

  // ---- RoPE table, built on the host in double, stored as fp32
  {
    const int half = c->d / 2;
    const size_t rows = (size_t)cfg->max_context;
    std::vector<float> cs(rows * half), sn(rows * half);
    for (size_t p = 0; p < rows; ++p)
      for (int i = 0; i < half; ++i) {
        double theta = (double)p * std::pow((double)cfg->rope_base, -2.0 * i / c->d);
        cs[p * half + i] = (float)std::cos(theta);
        sn[p * half + i] = (float)std::sin(theta);
      }
    size_t bytes = rows * half * 4;
    if (dev_malloc(&c->d_cos, bytes) != cudaSuccess || dev_malloc(&c->d_sin, bytes) != cudaSuccess) {
      fail(c, MAG_ERR_OOM, "RoPE table");
      return bail(MAG_ERR_OOM);
    }
    cudaMemcpy(c->d_cos, cs.data(), bytes, cudaMemcpyHostToDevice);
    cudaMemcpy(c->d_sin, sn.data(), bytes, cudaMemcpyHostToDevice);
    c->other_bytes += 2 * bytes + tb;
  }

  // ---- launch plans and arena
  {
    std::string why;
    if (!gemv_plans_fit(c, why)) {
      fail(c, MAG_ERR_INVALID_ARG, "create: %s", why.c_str());
      return bail(MAG_ERR_INVALID_ARG);
    }
  }
  build_decode_plan(c);
  if ((e = dev_malloc(&c->arena, std::max<uint64_t>(c->arena_bytes, 256))) != cudaSuccess) {
    fail(c, MAG_ERR_OOM, "arena: %s", cudaGetErrorString(e));
    return bail(MAG_ERR_OOM);
  }
  if (c->canary_band) cudaMemsetAsync(c->arena, kCanaryByte, c->arena_bytes, c->stream);
  c->r = (float*)arena_ptr(c, "residual");
  c->ss_part = (float*)arena_ptr(c, "sumsq_part");
  c->qkv = (__half*)arena_ptr(c, "qkv");
  c->o = (__half*)arena_ptr(c, "attn_out");
  c->act = (__half*)arena_ptr(c, "ffn_act");
  c->gemv_part = (float*)arena_ptr(c, "gemv_partial");

  // ---- counters, step arguments, staging
  size_t nc = gemv_counters(c);
  c->n_counters = nc;
  size_t stage_out = (size_t)c->B_max * (c->V ? c->V : c->D) * 2;
  const size_t part_bytes = (size_t)c->B_max * c->Hkv * kAttnMaxGroups * 3 * c->Hq / c->Hkv * c->d * 4;
  const size_t arrival_bytes = (size_t)c->B_max * c->Hkv * 4;
  if (dev_malloc(&c->d_counters, nc * 4) != cudaSuccess ||
      dev_malloc(&c->attn_part, part_bytes) != cudaSuccess ||
      dev_malloc(&c->attn_arrivals, arrival_bytes) != cudaSuccess ||
      dev_malloc(&c->d_args, sizeof(StepArgs)) != cudaSuccess ||
      dev_malloc(&c->d_in_stage, (size_t)c->B_max * c->D * 2) != cudaSuccess ||
      dev_malloc(&c->d_out_stage, stage_out) != cudaSuccess ||
      host_alloc(&c->h_ring, sizeof(StepArgs) * kRing, cudaHostAllocDefault) != cudaSuccess ||
      host_alloc(&c->h_err, sizeof(uint32_t), cudaHostAllocMapped) != cudaSuccess ||
      cudaHostGetDevicePointer(&c->d_err, c->h_err, 0) != cudaSuccess) {
    fail(c, MAG_ERR_OOM, "counters / step arguments");
    return bail(MAG_ERR_OOM);
  }
  *c->h_err = 0;
  if (cfg->max_chunk > 0) {
    mag_status ps = setup_prefill(c);
    if (ps != MAG_OK) return bail(ps);
  }
  cudaMemsetAsync(c->d_counters, 0, nc * 4, c->stream);
  cudaMemsetAsync(c->attn_arrivals, 0, arrival_bytes, c->stream);
  c->other_bytes += part_bytes + arrival_bytes;
  for (auto& ev : c->ring_ev) cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
  for (auto& ev : c->ev_step) cudaEventCreate(&ev);
  c->other_bytes += nc * 4 + sizeof(StepArgs) + (size_t)c->B_max * c->D * 2 + stage_out;
  if ((e = cudaStreamSynchronize(c->stream)) != cudaSuccess) {
    fail(c, MAG_ERR_CUDA, "create: %s", cudaGetErrorString(e));
    return bail(MAG_ERR_CUDA);
  }
  *out = c;
  return MAG_OK;
}

void mag_destroy(mag_ctx* c) { free_ctx(c); }

const char* mag_last_error(mag_ctx* c) { return c ? c->err.c_str() : "null context"; }

uint64_t mag_kv_bytes_per_token(const mag_config* g) {
  if (!g || g->head_dim <= 0) return 0;
  return 2ull * g->n_layers * g->n_kv_heads *
         (uint64_t)(kv_data_bytes(g->head_dim, g->kv_dtype) + kv_meta_bytes(g->head_dim, g->kv_dtype));
}

mag_status mag_quantize_w4g32(const void* src, int64_t rows, int64_t cols, void* codes, void* sm, void* stream) {
  if (rows < 0 || cols <= 0 || (rows && (!src || !codes || !sm))) return MAG_ERR_INVALID_ARG;
  cudaError_t e = launch_quantize_w4g32((cudaStream_t)stream, (const float*)src, rows, cols, (uint8_t*)codes,
                                        (__half2*)sm);
  return e == cudaSuccess ? MAG_OK : MAG_ERR_CUDA;
}

mag_status mag_load_weights(mag_ctx* c, int32_t tensor, int32_t layer, const void* src, int32_t fmt, size_t bytes) {
  if (!c) return MAG_ERR_INVALID_ARG;
  if (!src) return fail(c, MAG_ERR_INVALID_ARG, "load_weights: null source");
  const bool per_layer = tensor >= MAG_W_QKV && tensor <= MAG_NORM_FFN;
  if (tensor < 0 || tensor > MAG_LM_HEAD) return fail(c, MAG_ERR_INVALID_ARG, "load_weights: bad tensor %d", tensor);
  if (per_layer && (layer < 0 || layer >= c->L))
    return fail(c, MAG_ERR_INVALID_ARG, "load_weights: bad layer %d", layer);
  if (tensor <= MAG_W_DOWN) {
    Proj& p = c->proj[(size_t)layer * 4 + tensor];
    if (fmt == MAG_FMT_F32_DENSE) {
      if (bytes != (size_t)p.N * p.K * 4)
        return fail(c, MAG_ERR_INVALID_ARG, "load_weights: %zu bytes, expected fp32 [%d, %d]", bytes, p.N, p.K);
      // quantise into a stream-ordered scratch copy in W4G32 bytes, then tile it
      uint8_t* canon = nullptr;
      cudaError_t ea = dev_malloc_async(reinterpret_cast<void**>(&canon), p.canon_bytes, c->stream);
      if (ea == cudaErrorMemoryAllocation)
        return fail(c, MAG_ERR_OOM, "load_weights: %zu bytes of quantisation scratch: %s", p.canon_bytes,
                    cudaGetErrorString(ea));
      CUDA_TRY(c, ea);
      cudaError_t e1 = launch_quantize_w4g32(c->stream, (const float*)src, p.N, p.K, canon,
                                             reinterpret_cast<__half2*>(canon + (size_t)p.N * p.G * 16));
      cudaError_t e2 = e1 == cudaSuccess ? launch_w4_to_tiles(c->stream, canon, p.N, p.K, p.map, p.map_arg, p.tiles)
                                         : e1;
      cudaError_t e3 = cudaFreeAsync(canon, c->stream);
      if (e2 != cudaSuccess || e3 != cudaSuccess)
        return fail(c, MAG_ERR_CUDA, "load_weights: %s", cudaGetErrorString(e2 != cudaSuccess ? e2 : e3));
    } else if (fmt == MAG_FMT_W4G32) {
      if (bytes != p.canon_bytes)
        return fail(c, MAG_ERR_INVALID_ARG, "load_weights: %zu bytes, expected W4G32 %zu", bytes, p.canon_bytes);
      CUDA_TRY(c, launch_w4_to_tiles(c->stream, (const uint8_t*)src, p.N, p.K, p.map, p.map_arg, p.tiles));
    } else {
      return fail(c, MAG_ERR_INVALID_ARG, "load_weights: projections take FP32_DENSE or W4G32");
    }
    c->loaded[(size_t)layer * 6 + tensor] = 1;
    return MAG_OK;
  }
  if (fmt != MAG_FMT_F16) return fail(c, MAG_ERR_INVALID_ARG, "load_weights: norms and LM head take F16");
  if (tensor == MAG_LM_HEAD) {
    if (!c->V) return fail(c, MAG_ERR_INVALID_ARG, "load_weights: this model has no LM head");
    if (bytes != (size_t)c->V * c->D * 2) return fail(c, MAG_ERR_INVALID_ARG, "load_weights: LM head size");
    CUDA_TRY(c, launch_f16_to_tiles(c->stream, (const __half*)src, c->V, c->D, reinterpret_cast<uint8_t*>(c->lm_head)));
    c->loaded[(size_t)c->L * 6 + 1] = 1;
    return MAG_OK;
  }
  if (bytes != (size_t)c->D * 2) return fail(c, MAG_ERR_INVALID_ARG, "load_weights: norm gain size");
  __half* dst = tensor == MAG_NORM_ATTN ? c->gamma1[layer] : (tensor == MAG_NORM_FFN ? c->gamma2[layer] : c->gamma_f);
  CUDA_TRY(c, cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, c->stream));
  if (tensor == MAG_NORM_FINAL) c->loaded[(size_t)c->L * 6] = 1;
  else c->loaded[(size_t)layer * 6 + tensor] = 1;
  return MAG_OK;
}

mag_status mag_load_weights_f32_noalloc(mag_ctx* c, int32_t tensor, int32_t layer, const void* src, size_t bytes) {
  if (!c) return MAG_ERR_INVALID_ARG;
  if (!src) return fail(c, MAG_ERR_INVALID_ARG, "load_weights_f32_noalloc: null source");
  if (tensor < MAG_W_QKV || tensor > MAG_W_DOWN)
    return fail(c, MAG_ERR_INVALID_ARG, "load_weights_f32_noalloc: tensor %d is not a projection", tensor);
  if (layer < 0 || layer >= c->L) return fail(c, MAG_ERR_INVALID_ARG, "load_weights_f32_noalloc: bad layer %d", layer);
  Proj& p = c->proj[(size_t)layer * 4 + tensor];
  if (bytes != (size_t)p.N * p.K * 4)
    return fail(c, MAG_ERR_INVALID_ARG, "load_weights_f32_noalloc: %zu bytes, expected fp32 [%d, %d]", bytes, p.N,
                p.K);
  if (noalloc_slab_tiles(p.K, p.map, p.map_arg) == 0)
    return fail(c, MAG_ERR_INVALID_ARG,
                "load_weights_f32_noalloc: rows of %d values need more than the %zu-byte scratch per slab", p.K,
                kNoAllocScratchBytes);
  int dev = -1;
  CUDA_TRY(c, cudaGetDevice(&dev));
  if (dev != c->device)
    return fail(c, MAG_ERR_INVALID_ARG, "load_weights_f32_noalloc: make the context's device %d current (not %d)",
                c->device, dev);
  CUDA_TRY(c, load_f32_noalloc(c->stream, (const float*)src, p.N, p.K, p.map, p.map_arg, p.tiles));
  c->loaded[(size_t)layer * 6 + tensor] = 1;
  return MAG_OK;
}

mag_status mag_session_open(mag_ctx* c, int32_t* sid) {
  if (!c || !sid) return MAG_ERR_INVALID_ARG;
  for (size_t i = 0; i < c->sessions.size(); ++i)
    if (!c->sessions[i].open) {
      c->sessions[i].open = true;
      c->sessions[i].len = 0;
      c->sessions[i].table.clear();
      *sid = (int32_t)i;
      return MAG_OK;
    }
  return fail(c, MAG_ERR_INVALID_ARG, "session_open: all %d sessions are open", (int)c->sessions.size());
}

mag_status mag_session_close(mag_ctx* c, int32_t sid) {
  if (!c) return MAG_ERR_INVALID_ARG;
  if (sid < 0 || sid >= (int)c->sessions.size() || !c->sessions[sid].open)
    return fail(c, MAG_ERR_INVALID_ARG, "session_close: session %d is not open", sid);
  for (int32_t b : c->sessions[sid].table) c->kv.push(b);
  c->sessions[sid] = Session();
  return pool_trim(c);
}

mag_status mag_session_length(mag_ctx* c, int32_t sid, int32_t* len) {
  if (!c || !len) return MAG_ERR_INVALID_ARG;
  if (sid < 0 || sid >= (int)c->sessions.size() || !c->sessions[sid].open)
    return fail(c, MAG_ERR_INVALID_ARG, "session %d is not open", sid);
  *len = c->sessions[sid].len;
  return MAG_OK;
}

mag_status mag_kv_append(mag_ctx* c, int32_t sid, int32_t n, const void* k, const void* v) {
  if (!c) return MAG_ERR_INVALID_ARG;
  if (sid < 0 || sid >= (int)c->sessions.size() || !c->sessions[sid].open)
    return fail(c, MAG_ERR_INVALID_ARG, "kv_append: session %d is not open", sid);
  if (n < 0 || (n > 0 && (!k || !v))) return fail(c, MAG_ERR_INVALID_ARG, "kv_append: bad arguments");
  Session& s = c->sessions[sid];
  if ((int64_t)s.len + n > c->cfg.max_context)
    return fail(c, MAG_ERR_CONTEXT_FULL, "kv_append: %d + %d tokens exceed max_context %d", s.len, n,
                c->cfg.max_context);
  const int nb_old = (s.len + 15) / 16, nb_new = (s.len + n + 15) / 16;
  if (n == 0) return MAG_OK;
  mag_status st = reserve_blocks(c, "kv_append", nb_new - nb_old);
  if (st != MAG_OK) return st;
  for (int i = nb_old; i < nb_new; ++i) s.table.push_back(c->kv.pop());
  int32_t* row = c->d_tables + (size_t)sid * c->table_stride;
  if (nb_new > nb_old)
    CUDA_TRY(c, cudaMemcpyAsync(row + nb_old, s.table.data() + nb_old, (size_t)(nb_new - nb_old) * 4,
                                cudaMemcpyHostToDevice, c->stream));
  KvStoreArgs a = {};
  a.k = (const __half*)k;
  a.v = (const __half*)v;
  a.n_tok = n;
  a.n_layers = c->L;
  a.pos0 = s.len;
  a.table = row;
  a.pool = pool_geom(c);
  a.err = c->d_err;
  Launch L{c->stream, false, nullptr};
  // grid.x is the token count: split very long appends to respect the grid limit
  for (int t0 = 0; t0 < n; t0 += 65535) {
    KvStoreArgs b = a;
    b.n_tok = std::min(65535, n - t0);
    b.pos0 = s.len + t0;
    // the source is [L][n][Hkv][d]: a slice of tokens is strided per layer, so
    // slices go one layer at a time
    for (int l = 0; l < c->L; ++l) {
      KvStoreArgs bl = b;
      bl.k = a.k + ((size_t)l * n + t0) * c->Hkv * c->d;
      bl.v = a.v + ((size_t)l * n + t0) * c->Hkv * c->d;
      bl.n_layers = 1;
      bl.pool.base = c->kv.base() + (size_t)l * c->cfg.pool_blocks * c->block_bytes;
      CUDA_TRY(c, launch_kv_store(L, bl));
    }
  }
  s.len += n;
  return MAG_OK;
}

mag_status mag_sync(mag_ctx* c) {
  if (!c) return MAG_ERR_INVALID_ARG;
  CUDA_TRY(c, cudaStreamSynchronize(c->stream));
  return check_err(c);
}

mag_status mag_get_memory_stats(mag_ctx* c, mag_memory_stats* s) {
  if (!c || !s) return MAG_ERR_INVALID_ARG;
  memset(s, 0, sizeof *s);
  s->weight_bytes = c->wbytes;
  s->kv_pool_bytes = c->kv.reserved_bytes();
  s->kv_block_bytes = c->block_bytes;
  s->pool_blocks_total = c->cfg.pool_blocks;
  s->pool_blocks_free = (int32_t)c->kv.available();
  s->kv_pool_mapped_bytes = c->kv.mapped_bytes();
  s->pool_blocks_mapped = (int32_t)c->kv.mapped_blocks();
  s->pool_blocks_hot = (int32_t)c->kv.hot_blocks();
  s->pool_group_blocks = (int32_t)c->kv.group_blocks();
  s->arena_bytes = c->arena_bytes;
  s->arena_unshared_bytes = c->arena_unshared;
  s->other_device_bytes = c->other_bytes;
  s->prefill_weight_bytes = 0;  // the prefill GEMMs read the W4 tiles themselves
  s->prefill_arena_bytes = c->pf_arena_bytes;
  int open = 0;
  for (auto& x : c->sessions) open += x.open;
  s->sessions_open = open;
  return MAG_OK;
}

mag_status mag_debug_read_weights(mag_ctx* c, int32_t tensor, int32_t layer, void* dst, size_t bytes) {
  if (!c || !dst) return MAG_ERR_INVALID_ARG;
  if (tensor < MAG_W_QKV || tensor > MAG_W_DOWN || layer < 0 || layer >= c->L)
    return fail(c, MAG_ERR_INVALID_ARG, "debug_read_weights: projections only");
  Proj& p = c->proj[(size_t)layer * 4 + tensor];
  if (bytes != p.canon_bytes)
    return fail(c, MAG_ERR_INVALID_ARG, "debug_read_weights: expected %zu bytes", p.canon_bytes);
  CUDA_TRY(c, launch_w4_from_tiles(c->stream, p.tiles, p.N, p.K, p.map, p.map_arg, (uint8_t*)dst));
  return MAG_OK;
}

mag_status mag_debug_kv_locate(mag_ctx* c, int32_t sid, int32_t layer, int32_t tok, int64_t out[5]) {
  if (!c || !out) return MAG_ERR_INVALID_ARG;
  if (sid < 0 || sid >= (int)c->sessions.size() || !c->sessions[sid].open || layer < 0 || layer >= c->L || tok < 0 ||
      tok >= c->sessions[sid].len)
    return fail(c, MAG_ERR_INVALID_ARG, "debug_kv_locate: bad session/layer/token");
  const int blk = c->sessions[sid].table[tok / 16], slot = tok % 16;
  const int64_t base = ((int64_t)layer * c->cfg.pool_blocks + blk) * c->block_bytes;
  const int64_t vec = (int64_t)(0) * 16 + slot;
  (void)vec;
  const int64_t data_part = (int64_t)c->Hkv * 16 * c->data_bytes, meta_part = (int64_t)c->Hkv * 16 * c->meta_bytes;
  // head 0; callers add head * 16 * bytes per vector
  out[0] = base + (int64_t)slot * c->data_bytes;
  out[1] = base + data_part + (int64_t)slot * c->data_bytes;
  out[2] = c->meta_bytes ? base + 2 * data_part + (int64_t)slot * c->meta_bytes : -1;
  out[3] = c->meta_bytes ? base + 2 * data_part + meta_part + (int64_t)slot * c->meta_bytes : -1;
  out[4] = blk;
  return MAG_OK;
}

mag_status mag_debug_pool(mag_ctx* c, void** p, uint64_t* bytes) {
  if (!c || !p || !bytes) return MAG_ERR_INVALID_ARG;
  *p = c->kv.base();
  *bytes = c->kv.reserved_bytes();
  return MAG_OK;
}

mag_status mag_debug_arena_plan(mag_ctx* c, int32_t phase, mag_arena_tensor* out, int32_t cap, int32_t* n_out,
                                uint64_t* arena_bytes) {
  if (!c || !n_out || !arena_bytes || cap < 0 || (cap && !out)) return MAG_ERR_INVALID_ARG;
  if (phase != 0) return fail(c, MAG_ERR_UNSUPPORTED, "debug_arena_plan: only the decode phase is planned");
  *n_out = (int32_t)c->plan.size();
  *arena_bytes = c->arena_bytes;
  for (int i = 0; i < (int)c->plan.size() && i < cap; ++i) {
    memset(&out[i], 0, sizeof out[i]);
    snprintf(out[i].name, sizeof out[i].name, "%s", c->plan[i].name.c_str());
    out[i].size = c->plan[i].size;
    out[i].first = c->plan[i].first;
    out[i].last = c->plan[i].last;
    out[i].offset = c->plan[i].offset;
  }
  return MAG_OK;
}

int32_t mag_debug_last_step_launches(mag_ctx* c) { return c ? c->last_launches : 0; }

mag_status mag_debug_set_table_entry(mag_ctx* c, int32_t sid, int32_t idx, int32_t value) {
  if (!c) return MAG_ERR_INVALID_ARG;
  if (sid < 0 || sid >= (int)c->sessions.size() || !c->sessions[sid].open)
    return fail(c, MAG_ERR_INVALID_ARG, "debug_set_table_entry: session %d is not open", sid);
  if (idx < 0 || idx >= (int)c->sessions[sid].table.size())
    return fail(c, MAG_ERR_INVALID_ARG, "debug_set_table_entry: index %d not in 0..%d", idx,
                (int)c->sessions[sid].table.size() - 1);
  CUDA_TRY(c, cudaMemcpyAsync(c->d_tables + (size_t)sid * c->table_stride + idx, &value, 4, cudaMemcpyHostToDevice,
                              c->stream));
  CUDA_TRY(c, cudaStreamSynchronize(c->stream));
  return MAG_OK;
}

mag_status mag_debug_arena(mag_ctx* c, void** p, uint64_t* bytes) {
  if (!c || !p || !bytes) return MAG_ERR_INVALID_ARG;
  *p = c->arena;
  *bytes = c->arena_bytes;
  return MAG_OK;
}

mag_status mag_get_step_stats(mag_ctx* c, mag_step_stats* out) {
  if (!c || !out) return MAG_ERR_INVALID_ARG;
  *out = c->stats;
  out->last_ms = -1.0;
  if (c->step_timed && c->stats.steps > 0) {
    CUDA_TRY(c, cudaEventSynchronize(c->ev_step[1]));
    float ms = 0.f;
    CUDA_TRY(c, cudaEventElapsedTime(&ms, c->ev_step[0], c->ev_step[1]));
    out->last_ms = ms;
  }
  return MAG_OK;
}

}  // extern "C"
