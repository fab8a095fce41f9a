// Host side of the decode-step library, shared by its C-ABI units: capi.cu (context, weights, sessions,
// KV pool, statistics, debug hooks), step.cu (the decode step, its graphs and the adaptive plans), prefill.cu
// (chunked prefill) and verify.cu (the verify step of speculative decoding).
#pragma once
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

namespace mag {

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

}  // namespace mag

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
  // step timeline (mag_debug_timeline): the record buffer the next launches stamp into (rec null: off)
  TraceBuf trace = {};
  unsigned int* trace_n = nullptr;
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
  uint64_t canary_band = 0;  // MAG_FLAG_DEBUG_CANARY: bytes of each band before and after an arena tensor
  // mag_get_step_stats: the last call's figures, and its event pair (MAG_FLAG_STEP_TIMING)
  mag_step_stats stats{};
  cudaEvent_t ev_step[2] = {nullptr, nullptr};
  bool step_timed = false;

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

namespace mag {

#define CUDA_TRY(ctx, call)                                                                         \
  do {                                                                                              \
    cudaError_t e_ = (call);                                                                        \
    if (e_ != cudaSuccess) return fail(ctx, MAG_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

inline size_t align256(size_t v) { return (v + 255) / 256 * 256; }

constexpr size_t kPipeBudget = 200 * 1024, kSmemMax = 227 * 1024;

mag_status fail(mag_ctx* c, mag_status s, const char* fmt, ...);
mag_status check_err(mag_ctx* c);
ArenaCheck arena_check_args(const mag_ctx* c);  // the decode arena's canary bands
GemvPlan plan_gemv(const mag_ctx* c, int kind, int n_mtiles, int K, int B);
int attn_splits(const mag_ctx* c, int B, bool wide = false);
PoolGeom pool_geom(const mag_ctx* c);
mag_status reserve_blocks(mag_ctx* c, const char* what, int64_t n);
bool group_referenced(const mag_ctx* c, int64_t g);
mag_status pool_trim(mag_ctx* c);
bool all_loaded(const mag_ctx* c);
// The decode step's projections: kind (0 QKV, 1 O, 2 gate-up, 3 down, 4 LM head), tiles, K, launch variant
struct ProjShape {
  int kind, n_mtiles, K, wfmt, xsrc, epi;
};
std::vector<ProjShape> proj_shapes(const mag_ctx* c);
size_t gemv_partial_floats(const mag_ctx* c, int B);
bool gemv_plans_fit(const mag_ctx* c, std::string& why);
size_t gemv_counters(const mag_ctx* c);
void build_decode_plan(mag_ctx* c);
void* arena_ptr(mag_ctx* c, const char* name);
GemvArgs gemv_args(const mag_ctx* c, int kind, const uint8_t* w, int n_mtiles, int K, int B);
void free_ctx(mag_ctx* c);
mag_status check_cfg(const mag_config* g, std::string& why);

// step.cu
cudaError_t record_step(mag_ctx* c, int B, int* n_launch, Profiler* prof, bool verify, int splits, bool wide,
                        cudaStream_t st, float* resid_dump = nullptr);
mag_status step_prepare(mag_ctx* c, int B, const int32_t* sids, StepArgs& a);
mag_status step_upload(mag_ctx* c, int B, const int32_t* sids, const void* in, void* out);
bool plan_wide(const mag_ctx* c, int p);
int plan_splits(const mag_ctx* c, int p, int B);
struct AttnShape {
  int splits;
  bool wide;
  int bucket;  // -1: the adaptive plan's graphs
};
AttnShape attn_shape(const mag_ctx* c, int B);
mag_status poll_capture(mag_ctx* c);
mag_status finish_capture(mag_ctx* c);
void switch_plan(mag_ctx* c, int p);
void adapt_after_step(mag_ctx* c, int B, const int32_t* lens);
mag_status launch_step(mag_ctx* c, int B, bool verify);
// statistics of a call about to launch: kind (0 decode, 1 verify step, 2 chunk path), rows, the keys each
// row attends; records the start event with MAG_FLAG_STEP_TIMING
mag_status stats_begin(mag_ctx* c, int kind, int rows, int out_rows, const int32_t* keys, int n_keys_rows);
mag_status stats_end(mag_ctx* c);  // launches from last_launches; the end event

// prefill.cu
mag_status setup_prefill(mag_ctx* c);
mag_status run_chunk(mag_ctx* c, const char* what, int n_seg, const int32_t* sids, const int32_t* ntok,
                     const void* in, void* out, bool all_rows, float* resid_dump = nullptr);

}  // namespace mag
