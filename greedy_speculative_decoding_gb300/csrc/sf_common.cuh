// Shared device helpers and kernel parameter blocks of the engine.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sf.h"

namespace sf {

typedef __nv_bfloat16 bf16;

constexpr int kRows = SF_MAX_ROWS;     // tokens per forward, at most
constexpr int kGroupRows = 16;         // token rows of one GEMM CTA (a forward of more rows runs
                                       // ceil(M / 16) row groups side by side)
constexpr int kMaxGroups = kRows / kGroupRows;
constexpr int kBlockRows = 128;        // output rows (features) per GEMM CTA
constexpr int kGemmThreads = 256;      // 8 warps x 16 rows
constexpr int kChunk = 64;             // k per pipeline step (one 128-byte line per weight row)
#ifndef SF_STAGES
#define SF_STAGES 4
#endif
constexpr int kStages = SF_STAGES;          // weight tiles in flight per warp (TMA ring)
constexpr int kTileBytes = 16 * kChunk * 2;   // one warp's 16 rows x 64 k of bf16
constexpr int kKvChunk = 64;           // cache slots per attention work item
constexpr int kAttnThreads = 256;

// Device error bits (engine status word).
constexpr int kErrNonfinite = 1;
constexpr int kErrWait = 2;
constexpr int kErrCapacity = 4;

// Rows of one forward: row m belongs to sequence m / rps and sits in cache
// slot pos_base[m / rps] + pos_off + m % rps. That slot is also its sequence
// position, except in a verify pass over several candidate guesses
// (tree_g = g > 0): there row j >= 1 of a sequence is guess (j - 1) % g of
// candidate (j - 1) / g, at position p0 + 1 + (j - 1) % g (p0: row 0's slot),
// and it sees the slots up to p0 and its own candidate's slots up to itself.
struct RowSet {
  const int* tok;      // token of row m: tok[b * tok_stride + tok_off + j]
  int tok_stride, tok_off;
  int rps;             // rows per sequence
  int M;               // rows in total
  const int* pos_base;
  int pos_off;
  unsigned long long* trace;   // optional launch timeline: [2 * trace_id + {0: entry, 1: producer done}]
  int trace_id;
  int tree_g;          // guesses per candidate of a multi-candidate verify pass; 0: one chain
};

constexpr int kTraceSlots = 8192;   // launch timeline slots (ring)

// Launch timeline for profiling: CTA 0 stamps the global timer when the
// kernel starts and when its wait on the preceding kernel returns (that is,
// when the preceding kernel has finished).
__device__ __forceinline__ void trace_mark(const RowSet& rs, int k) {
  if (rs.trace && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    rs.trace[2 * rs.trace_id + k] = t;
  }
}

// One weight-side scalar (gain, bias, embedding entry): bf16, or fp32.
__device__ __forceinline__ float ldw(const void* p, size_t i, int f32) {
  return f32 ? static_cast<const float*>(p)[i] : __bfloat162float(static_cast<const bf16*>(p)[i]);
}

// Set an error bit in the caller's status word; launches made outside an
// engine (sf_linear) carry no status word and report nothing.
__device__ __forceinline__ void report_err(int* err, int bit) {
  if (err) atomicOr(err, bit);
}

__device__ __forceinline__ int row_slot(const RowSet& rs, int m) {
  return rs.pos_base[m / rs.rps] + rs.pos_off + m % rs.rps;
}
// Slots between row 0 and row j's own candidate: (j - 1) / g * g of them.
__device__ __forceinline__ int tree_gap(const RowSet& rs, int j) {
  return (rs.tree_g > 0 && j > 0) ? (j - 1) / rs.tree_g * rs.tree_g : 0;
}
// Sequence position of row m (its RoPE angle).
__device__ __forceinline__ int row_pos(const RowSet& rs, int m) {
  return row_slot(rs, m) - tree_gap(rs, m % rs.rps);
}

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Bounded wait on an mbarrier phase. Returns false if it gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t max_iter) {
  uint32_t addr = smem_u32(bar);
  for (uint32_t it = 0; it < max_iter; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// Two-dimensional tensor tile global -> shared (TMA) at coordinates (x, y),
// completion on an mbarrier, with an L2 eviction-priority policy.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// For weight tiles that other row groups of the same launch read again.
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 16-byte asynchronous global -> shared copy (LDGSTS), its group commit and wait.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Thread-block clusters: full-cluster barrier (release/acquire), this CTA's
// rank, and loads from another CTA's shared memory (distributed shared memory).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The two halves of that barrier, for work between arriving and waiting.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
// Arrival that publishes nothing (the caller's shared memory is not read by
// the other CTAs after this barrier phase).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local_smem, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_smem), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ float ld_dsmem(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// 16-byte asynchronous store into another CTA's shared memory (cluster
// address), counted in bytes on that CTA's mbarrier (cluster address).
__device__ __forceinline__ void st_async_v4(uint32_t addr, float4 v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   addr),
               "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
               : "memory");
}

// Bounded wait on an mbarrier phase completed by other CTAs of the cluster
// (acquire at cluster scope). Returns false if it gave up.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t max_iter) {
  const uint32_t addr = smem_u32(bar);
  for (uint32_t it = 0; it < max_iter; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// Programmatic dependent launch: wait for the preceding grid's results /
// allow the next grid to start its prologue.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_next() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(bf16 lo, bf16 hi) {
  return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}

// Order-preserving map of a float to an unsigned key (larger float -> larger key).
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Packed (value, index) key: larger value wins, then the lower index.
__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
  return ((unsigned long long)float_key(v) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}

__device__ __forceinline__ int key_index(unsigned long long k) {
  return (int)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
}

// ------------------------------------------------ fragment-ordered activations
// The GEMM's B operand (token activations) lives in global memory already in
// the order its warps read it: for T = ceil(M / 4) token tiles, 64-feature
// chunk j, tile t and half h (features 8h..8h+7 of each 16), lane l holds 8
// bf16 in 16 bytes at unit ((j * T + t) * 2 + h) * 32 + l. Lane l = 4 * col + c
// serves MMA column col = 2 * (m % 4) + {0: hi, 1: lo} of token m = 4t + m % 4
// and features k = 64j + 16c + 8h + e (e = 0..7). Each value is stored as a
// bf16 pair (hi = bf16(v), lo = bf16(v - hi)), so products keep about 16
// mantissa bits of the fp32 value. Bytes for K features: frag_bytes(K, T).
__host__ __device__ __forceinline__ size_t frag_bytes(int K, int T) {
  return (size_t)((K + 63) / 64) * T * 1024;
}

// bf16 index of the hi part of (token m, feature k); the lo part is 32 further.
__device__ __forceinline__ size_t frag_index(int m, int k, int T) {
  const int j = k >> 6, kk = k & 63;
  const int c = kk >> 4, h = (kk >> 3) & 1, e = kk & 7;
  const int t = m >> 2, col = 2 * (m & 3);
  return ((((size_t)j * T + t) * 2 + h) * 32 + 4 * col + c) * 8 + e;
}


// ------------------------------------------------ tensor-core operand order
// Forwards of more than 16 token rows run their projections on the tcgen05
// tensor cores, with the activations as plain bf16 (one operand row per
// token) in the MMA's canonical K-major B tile with 128-byte swizzle: for
// 64-feature chunk j and token tile t (tokens 8t .. 8t+7) one 1024-byte
// block at byte (j * T8 + t) * 1024, T8 = ceil(M / 8), holds 8 rows of 128
// bytes, row m % 8; the 16-byte piece with features 8q .. 8q+7 of the chunk
// sits at position q ^ (m % 8) of its row. A chunk of all T8 tiles is one
// contiguous T8 * 1024-byte block that a single bulk copy brings into shared
// memory ready for the MMA.
__device__ __forceinline__ size_t umma_index(int m, int k, int T8) {
  const int j = k >> 6, kk = k & 63;
  const int t = m >> 3, row = m & 7;
  const int q = kk >> 3, e = kk & 7;
  return (((size_t)j * T8 + t) * 1024 + row * 128 + ((q ^ row) << 4)) / 2 + e;
}

// Store one activation in the order its consumer reads: fragment order
// (mma.sync GEMMs: a bf16 hi/lo pair) or the tensor-core operand order (bf16).
// T = ceil(M / 4), the fragment layout's tile count.
__device__ __forceinline__ void act_store(bf16* f, int m, int k, int T, float v, int umma) {
  const bf16 hi = __float2bfloat16_rn(v);
  if (umma) {
    f[umma_index(m, k, (T + 1) >> 1)] = hi;
  } else {
    const size_t i = frag_index(m, k, T);
    f[i] = hi;
    f[i + 32] = __float2bfloat16_rn(v - __bfloat162float(hi));
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

}  // namespace sf
