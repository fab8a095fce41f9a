// C ABI of the decode-step library: context, weights, KV block pool, arena
// plan, CUDA-graph step and the debug hooks. See include/mag.h for the
// contract of each call.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <deque>
#include <memory>
#include <string>
#include <thread>
#include <vector>

#include "adapt.h"
#include "alloc.h"
#include "arena.h"
#include "kernels.h"
#include "kvpool.h"
#include "noalloc.h"
#include "mag.h"

using namespace mag;

namespace {

constexpr int kRing = 8;

struct Proj {
  uint8_t* tiles = nullptr;  // [N/16][ceil(K/64)][640 B]
  int N = 0, K = 0, G = 0;
  int map = 0, map_arg = 0;  // tile row map (TileMap) and its argument
  size_t canon_bytes = 0;    // W4G32 bytes: N * G * 20
  size_t tile_bytes = 0;
};

struct Session {
  bool open = false;
  int len = 0;
  std::vector<int32_t> table;
};

struct GemvPlan {
  int n_cta, stages, t_max;  // pipelined kernels (up to kPipeMaxBatch tokens; W4 above); n_cta = 0 otherwise
  int ks, cpc, tpw;          // k-ranges (W4 above kPipeMaxBatch: windows) and their chunks; fp16 k-split tpw
  size_t smem;
};

// Event pairs around each launch of an instrumented (eager) step.
struct Profiler {
  std::vector<cudaEvent_t> start, stop;
  std::vector<int> kinds;
  cudaError_t begin(cudaStream_t s) {
    cudaEvent_t e;
    cudaError_t r = cudaEventCreate(&e);
    if (r != cudaSuccess) return r;
    start.push_back(e);
    return cudaEventRecord(e, s);
  }
  cudaError_t end(cudaStream_t s, int kind) {
    cudaEvent_t e;
    cudaError_t r = cudaEventCreate(&e);
    if (r != cudaSuccess) return r;
    stop.push_back(e);
    kinds.push_back(kind);
    return cudaEventRecord(e, s);
  }
  ~Profiler() {
    for (auto e : start) cudaEventDestroy(e);
    for (auto e : stop) cudaEventDestroy(e);
  }
};

}  // namespace

struct mag_ctx {
  mag_config cfg{};
  cudaStream_t stream = nullptr;
  bool own_stream = false;
  int device = 0, n_sm = 0;
  int attn_cluster_max = 1;       // largest co-scheduled attention cluster, 4-warp blocks
  int attn_cluster_max_wide = 1;  // the same for the wide (16- or 8-warp) blocks
  float* attn_part = nullptr;       // clusters' partial outputs when a (session, KV head) spans several
  uint32_t* attn_arrivals = nullptr;
  std::string err;
  int L = 0, D = 0, Hq = 0, Hkv = 0, d = 0, F = 0, V = 0, R = 0, G = 0, B_max = 0;
  int table_stride = 0;

  // weights
  uint8_t* wbase = nullptr;
  size_t wbytes = 0;
  std::vector<Proj> proj;  // [L][4]
  std::vector<__half*> gamma1, gamma2;
  __half* gamma_f = nullptr;
  __half* lm_head = nullptr;
  std::vector<uint8_t> loaded;  // [L][6] + final norm + lm head

  // KV pool
  KvPool kv;  // memory and free list (fixed, or elastic hot / cold groups)
  int64_t block_bytes = 0;
  int data_bytes = 0, meta_bytes = 0;
  int32_t* d_tables = nullptr;
  std::vector<Session> sessions;

  // RoPE table
  float* d_cos = nullptr;
  float* d_sin = nullptr;

  // activation arena (decode phase)
  uint8_t* arena = nullptr;
  uint64_t arena_bytes = 0, arena_unshared = 0;
  std::vector<ArenaTensor> plan;
  float* r = nullptr;
  __half* qkv = nullptr;
  __half* o = nullptr;
  float* ss_part = nullptr;
  __half* act = nullptr;
  float* gemv_part = nullptr;

  // counters (zero between launches) and step arguments
  uint32_t* d_counters = nullptr;
  uint32_t* h_err = nullptr;  // mapped pinned word: kernels set bits when a bounded wait gives up
  uint32_t wait_limit = kWaitPolls;  // polls of a GEMV main-loop wait (mag_debug_set_wait_limit)
  uint32_t* d_err = nullptr;
  size_t n_counters = 0;
  StepArgs* d_args = nullptr;
  StepArgs* h_ring = nullptr;
  cudaEvent_t ring_ev[kRing] = {};
  int ring_pos = 0;

  // staging for the host-buffer step
  void* d_in_stage = nullptr;
  void* d_out_stage = nullptr;

  // captured step graphs by [verify][plan][batch]: a verify step's rows are the drafts of one session
  struct StepGraph {
    cudaGraphExec_t exec = nullptr;
    int launches = 0;
  };
  StepGraph graphs[2][3][MAG_MAX_BATCH + 1];
  // without the adaptive runtime: graphs by [verify][context bucket][batch] (attention splits by the step's
  // longest context)
  static constexpr int kLenBuckets = 4;
  StepGraph len_graphs[2][kLenBuckets][MAG_MAX_BATCH + 1];
  int step_max_len = 0;  // longest context (position + 1) among the rows of the step being launched
  int last_launches = 0;

  // adaptive runtime: load profile, plan in use, background capture of a new plan's graphs
  mag_adapt_config adapt{};  // enable_adaptive = 0 until mag_set_adaptive
  std::unique_ptr<LoadProfile> profile;
  int cur_plan = 1;
  int switches = 0;
  int64_t hot_blocks = -1;
  int pending_plan = -1;
  std::thread cap_thread;
  std::atomic<int> cap_state{0};  // 0 idle, 1 capturing, 2 done, 3 failed
  std::string cap_err;
  cudaStream_t cap_stream = nullptr;
  uint64_t other_bytes = 0;
  // chunked prefill (max_chunk > 0): planned buffers and the activations' TMA maps (the GEMMs read the W4 tiles)
  uint8_t* pf_arena = nullptr;
  uint64_t pf_arena_bytes = 0;
  std::vector<ArenaTensor> pf_plan;
  float* pf_r = nullptr;
  __half* pf_xn = nullptr;
  __half* pf_qkv = nullptr;
  __half* pf_o = nullptr;
  __half* pf_act = nullptr;
  int32_t* pf_rows = nullptr;   // [2][max_chunk]: position and session of every row (several sessions)
  float* pf_part = nullptr;     // split-K GEMMs: partial sums of the two K halves
  uint32_t* pf_part_cnt = nullptr;
  float* pf_last_r = nullptr;   // [MAG_MAX_BATCH][D]: the sessions' last residual rows, gathered
  alignas(64) uint8_t map_xn[128];
  alignas(64) uint8_t map_o[128];
  alignas(64) uint8_t map_act[128];
};

namespace {

mag_status fail(mag_ctx* c, mag_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (c) c->err = buf;
  return s;
}

#define CUDA_TRY(ctx, call)                                                                         \
  do {                                                                                              \
    cudaError_t e_ = (call);                                                                        \
    if (e_ != cudaSuccess) return fail(ctx, MAG_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// After a synchronisation: a kernel whose bounded wait gave up left a bit in the error word.
// The arrival counters of the last-to-arrive merges (GEMV tiles, attention clusters, prefill split-K) may be
// left part-way by a role that gave up: they start again from zero.
mag_status check_err(mag_ctx* c) {
  const uint32_t e = *reinterpret_cast<volatile uint32_t*>(c->h_err);
  if (e == 0) return MAG_OK;
  *reinterpret_cast<volatile uint32_t*>(c->h_err) = 0;
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
constexpr size_t kPipeBudget = 200 * 1024, kSmemMax = 227 * 1024;

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
int attn_splits(const mag_ctx* c, int B, bool wide = false) {
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

// The decode step's projections: kind (0 QKV, 1 O, 2 gate-up, 3 down, 4 LM head), tiles, K, launch variant
struct ProjShape {
  int kind, n_mtiles, K, wfmt, xsrc, epi;
};
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
  c->arena_bytes = plan_arena(c->plan, 64, (c->cfg.flags & MAG_FLAG_ARENA_NO_REUSE) != 0);
}

void* arena_ptr(mag_ctx* c, const char* name) {
  for (auto& t : c->plan)
    if (t.name == name) return c->arena + t.offset;
  return nullptr;
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
  return a;
}

// Enqueue the whole decode step for batch B (captured into a graph or run eagerly).
// The decode step's launches. With `verify` the B rows are B consecutive new tokens of one session: their
// keys and values go into the pool in one store kernel after the QKV projection, and attention reads them
// there (row b causally up to its own position) instead of each row appending its own.
// `splits` is the attention split count of the plan in use; `st` the stream the launches go to (the
// context's, or a capture stream). With `resid_dump` (eager debug steps only) the fp32 residual of the B rows
// is copied there after the step prologue and after every layer: [L+1][B][D].
cudaError_t record_step(mag_ctx* c, int B, int* n_launch, Profiler* prof, bool verify, int splits, bool wide,
                        cudaStream_t st, float* resid_dump = nullptr) {
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
#undef MAG_RUN
  return cudaSuccess;
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
  cudaFree(c->wbase);
  cudaFree(c->d_tables);
  cudaFree(c->d_cos);
  cudaFree(c->d_sin);
  cudaFree(c->arena);
  cudaFree(c->d_counters);
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

}  // namespace

namespace {

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

}  // namespace

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

static mag_status step_prepare(mag_ctx* c, int B, const int32_t* sids, StepArgs& a) {
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

static mag_status step_upload(mag_ctx* c, int B, const int32_t* sids, const void* in, void* out) {
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
static bool plan_wide(const mag_ctx* c, int p) { return c->adapt.enable_adaptive && c->adapt.plan_wide[p]; }

// Attention split count of plan p at batch B: the plan's count (a single-session figure), capped at about
// 4 blocks per SM over the batch's (session, KV head) pairs; 0 = the context's default (at most one
// cluster).
static int plan_splits(const mag_ctx* c, int p, int B) {
  const int s = c->adapt.enable_adaptive ? c->adapt.plan_splits[p] : 0;
  if (s == 0) return attn_splits(c, B, plan_wide(c, p));
  return std::max(1, std::min(s, 4 * c->n_sm / (B * c->Hkv)));
}

// Attention launch shape of the step being launched: the plan's with the adaptive runtime on; otherwise by
// the step's longest context, about 76 pool blocks per split (measured on GB300: 16 splits, one cluster, up
// to ~19k keys; 32 at ~39k; 64 at ~78k), so that long contexts keep enough warps streaming the pool.
struct AttnShape {
  int splits;
  bool wide;
  int bucket;  // -1: the adaptive plan's graphs
};
static AttnShape attn_shape(const mag_ctx* c, int B) {
  if (c->adapt.enable_adaptive) return {plan_splits(c, c->cur_plan, B), plan_wide(c, c->cur_plan), -1};
  const int nb = (c->step_max_len + 15) / 16, def = attn_splits(c, B);
  const int bk = nb <= 16 * 76 ? 0 : (nb <= 32 * 76 ? 1 : (nb <= 48 * 76 ? 2 : 3));
  const int s = bk == 0 ? def : std::max(def, std::min(16 * (bk + 1), 4 * c->n_sm / (B * c->Hkv)));
  return {s, false, bk};
}

// Capture and instantiate the step graph of (verify, plan p, batch B) on stream st: the context's
// stream, or the capture stream of a background switch.
static cudaError_t capture_graph(mag_ctx* c, bool verify, int p, int B, cudaStream_t st,
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
static mag_status poll_capture(mag_ctx* c) {
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
static mag_status finish_capture(mag_ctx* c) {
  if (c->cap_thread.joinable()) c->cap_thread.join();
  return poll_capture(c);
}

// Switch to plan p: at once (its graphs are captured on first use by the step), or, with async_switch,
// after a background thread has captured p's graphs for every shape the current plan has captured.
static void switch_plan(mag_ctx* c, int p) {
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
static void adapt_after_step(mag_ctx* c, int B, const int32_t* lens) {
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
static mag_status launch_step(mag_ctx* c, int B, bool verify) {
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

mag_status mag_decode_step(mag_ctx* c, int32_t B, const int32_t* sids, const void* in, void* out) {
  if (!c) return MAG_ERR_INVALID_ARG;
  mag_status st = poll_capture(c);
  if (st != MAG_OK) return st;
  st = step_upload(c, B, sids, in, out);
  if (st != MAG_OK) return st;
  st = launch_step(c, B, false);
  if (st != MAG_OK) return st;
  int32_t lens[MAG_MAX_BATCH];
  for (int b = 0; b < B; ++b) lens[b] = ++c->sessions[sids[b]].len;
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

namespace {

// The chunk path of mag_prefill_chunk and mag_verify_tokens: T tokens of one session through every layer
// (their k and v appended to the pool), then the final RMSNorm + LM head (or the final hidden state) of the
// last out_rows tokens into out [out_rows][V or D].
// One prefill chunk of n_seg sessions: session sids[i] appends ntok[i] tokens, the rows of the sessions
// following each other in `in` ([sum ntok][D]); each session's tokens attend causally to its own cache.
// Output: with all_rows (one session), every row; otherwise the last row of every session, in order.
// With resid_dump (debug) the launches run without programmatic dependent launch and the fp32 residual of
// the T rows is copied there after the input and after every layer: [L+1][T][D].
mag_status run_chunk(mag_ctx* c, const char* what, int n_seg, const int32_t* sids, const int32_t* ntok,
                     const void* in, void* out, bool all_rows, float* resid_dump = nullptr) {
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
  // step arguments of the output rows' LM head (or final hidden state)
  const int slot = c->ring_pos;
  CUDA_TRY(c, cudaEventSynchronize(c->ring_ev[slot]));
  StepArgs& sa = c->h_ring[slot];
  memset(&sa, 0, sizeof sa);
  sa.batch = out_rows;
  sa.out = out;
  PrefillAttnArgs pa = {};
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
  return MAG_OK;
}

}  // namespace

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
  st = launch_step(c, n, true);
  if (st != MAG_OK) return st;
  int32_t lens[MAG_MAX_BATCH];
  for (int b = 0; b < n; ++b) lens[b] = s.len + b + 1;
  s.len += n;
  adapt_after_step(c, n, lens);
  return pool_trim(c);
}

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

}  // extern "C"
