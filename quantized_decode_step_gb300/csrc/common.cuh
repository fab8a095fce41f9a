// Shared device helpers and launch-argument structs of the decode-step kernels.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define MAG_MAX_BATCH 16

// Error-word bits of the device-side checks (the waits that give up use bits 2-8): a pool block id read
// from a block table outside the pool (the id is not used), and a changed arena canary band (bit 16 + i:
// arena tensor i).
constexpr uint32_t kErrBounds = 2048u;
constexpr uint32_t kErrCanary = 1024u;
constexpr int kErrCanaryShift = 16;
// A pool block id from a block table, checked against the pool: an id outside it becomes 0 (a valid block)
// and sets kErrBounds.
__device__ __forceinline__ int checked_block(int phys, int pool_blocks, uint32_t* err) {
  if ((unsigned)phys < (unsigned)pool_blocks) return phys;
  if (err) atomicOr(err, kErrBounds);
  return 0;
}

// Step arguments uploaded once per decode step (one small H2D copy) and read
// by the kernels of the captured graph, so the graph itself never changes.
struct StepArgs {
  const __half* hidden_in;  // [B][D] fp16, caller owned
  void* out;                // [B][V] fp16 logits or [B][D] fp16 hidden, caller owned
  int32_t batch;
  int32_t n_upd;                    // block-table entries to write before the step
  int32_t sess[MAG_MAX_BATCH];      // session id of batch row b
  int32_t pos[MAG_MAX_BATCH];       // position of the new token = prior length
  int32_t upd_sess[MAG_MAX_BATCH];  // block-table writes: table[upd_sess][upd_idx] = upd_blk
  int32_t upd_idx[MAG_MAX_BATCH];
  int32_t upd_blk[MAG_MAX_BATCH];
  int32_t blk[MAG_MAX_BATCH];       // physical pool block of row b's new token (table[sess[b]][pos[b] / 16])
};

// KV pool geometry (block-major: (layer * P + block) * block_bytes, then
// K data [Hkv][16][d], V data, K meta [Hkv][16], V meta).
struct PoolGeom {
  uint8_t* base;
  int64_t block_bytes;
  int64_t pool_blocks;
  int32_t data_bytes;  // per (token, head) vector: 2d, d or d/2
  int32_t meta_bytes;  // per vector: 0, 2 or (d/32)*4
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t kv_dtype;
  const int32_t* tables;  // [max_sessions][table_stride] physical block ids
  int32_t table_stride;
};

__device__ __forceinline__ uint8_t* pool_vec(const PoolGeom& g, int layer, int blk, int part, int head, int slot) {
  int64_t base = ((int64_t)layer * g.pool_blocks + blk) * g.block_bytes;
  int64_t vec = (int64_t)head * 16 + slot;
  int64_t data_part = (int64_t)g.n_kv_heads * 16 * g.data_bytes;
  int64_t meta_part = (int64_t)g.n_kv_heads * 16 * g.meta_bytes;
  switch (part) {
    case 0: return g.base + base + vec * g.data_bytes;
    case 1: return g.base + base + data_part + vec * g.data_bytes;
    case 2: return g.base + base + 2 * data_part + vec * g.meta_bytes;
    default: return g.base + base + 2 * data_part + meta_part + vec * g.meta_bytes;
  }
}

// Step timeline (debug aid): with rec set, kernels append records of four u64 (tag, block (x | y << 20 |
// z << 40), event, %globaltimer in ns) at their phase boundaries; n counts the records attempted (those
// past cap are dropped). Passed in the kernels' arguments, so that a disabled timeline costs a parameter
// read per stamp point.
struct TraceBuf {
  unsigned long long* rec;
  unsigned int* n;
  unsigned int cap;
};
constexpr unsigned long long kTraceGemv = 1ull << 60, kTraceAttn = 2ull << 60;
__device__ __forceinline__ void trace_stamp(const TraceBuf& tb, unsigned long long tag, unsigned int ev) {
  if (!tb.rec) return;
  const unsigned int i = atomicAdd(tb.n, 1u);
  if (i >= tb.cap) return;
  unsigned long long ts;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(ts));
  ulonglong2* r = reinterpret_cast<ulonglong2*>(tb.rec + 4ull * i);
  r[0] = make_ulonglong2(tag, ((unsigned long long)blockIdx.z << 40) | ((unsigned long long)blockIdx.y << 20) |
                                  blockIdx.x);
  r[1] = make_ulonglong2(ev, ts);
}

// Programmatic dependent launch: wait for the producer grid's memory, and let
// the next grid's blocks start their prologue early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
  return d;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// D += A(16x16, row) * B(16x8, col), fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Streaming 64/128-bit loads of data read once per step.
__device__ __forceinline__ uint2 ldg_stream_u2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ldg_stream_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_nc_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
