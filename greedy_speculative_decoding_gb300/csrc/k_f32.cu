// Projections with fp32 weights (SF_WDTYPE_F32): the tiny correctness
// workload in single precision. Plain fp32 arithmetic on the CUDA cores (the
// model is a few MB; speed is not the point here), the same RMSNorm row
// factor and the same epilogues as the bf16 and NF4 kernels.
//
// One CTA per 128 output rows (SwiGLU: 64 gate rows, then the same features'
// 64 up rows) takes all of K and every token row: thread t owns output row
// t % 128 and the tokens of parity t / 128; each 64-feature chunk of the
// activations (read back from fragment order as hi + lo) is staged in shared
// memory and broadcast to the threads, each of which holds its row's 64
// weights in registers.
#include "gemm_epi.cuh"

namespace sf {

namespace {
constexpr int kF32Tok = (kRows + 1) / 2;   // tokens per thread (token parity)
}

template <int EPI>
__global__ void __launch_bounds__(kGemmThreads) k_gemm_f32(const __grid_constant__ GemmArgs a) {
  extern __shared__ float f32_smem[];
  float* ys = f32_smem;                        // [M][128]
  float* xs = ys + kRows * kBlockRows;         // [M][64] one chunk of activations
  __shared__ int s_pos[kRows];
  __shared__ float s_rinv[kRows];
  __shared__ int s_flag;
  trace_mark(a.rs, 0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int M = a.rs.M, T4 = (M + 3) / 4;
  const int rb = blockIdx.x;
  const int r = tid & (kBlockRows - 1), par = tid >> 7;
  // Weight row of output row r of this block.
  int seg, wrow;
  if (EPI == EPI_SWIGLU) {
    seg = r >> 6;
    wrow = rb * 64 + (r & 63);
  } else {
    const int n = rb * kBlockRows + r;
    seg = 0;
    while (seg < a.nseg - 1 && n >= a.seg_end[seg]) ++seg;
    wrow = n - (seg ? a.seg_end[seg - 1] : 0);
  }
  const int rows_seg = a.seg_end[seg] - (seg ? a.seg_end[seg - 1] : 0);
  const bool row_ok = EPI == EPI_SWIGLU ? wrow < a.N : wrow < rows_seg && rb * kBlockRows + r < a.N;
  const float* W = static_cast<const float*>(a.w[seg]) + (size_t)wrow * a.ld[seg];
  if (EPI == EPI_QKV && tid < M) s_pos[tid] = row_slot(a.rs, tid);
  pdl_wait();
  trace_mark(a.rs, 1);
  pdl_launch_next();

  float acc[kF32Tok];
#pragma unroll
  for (int i = 0; i < kF32Tok; ++i) acc[i] = 0.f;
  for (int k0 = 0; k0 < a.K; k0 += 64) {
    __syncthreads();   // the previous chunk's activations are consumed
    for (int i = tid; i < M * 64; i += kGemmThreads) {
      const int m = i >> 6, k = k0 + (i & 63);
      float v = 0.f;
      if (k < a.K) {
        const size_t fi = frag_index(m, k, T4);
        const bf16* in = reinterpret_cast<const bf16*>(a.in);
        v = __bfloat162float(in[fi]) + __bfloat162float(in[fi + 32]);
      }
      xs[i] = v;
    }
    float w[64];
#pragma unroll
    for (int k = 0; k < 64; ++k) w[k] = (row_ok && k0 + k < a.K) ? W[k0 + k] : 0.f;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kF32Tok; ++i) {
      const int m = par + 2 * i;
      if (m >= M) break;
      const float* xm = xs + m * 64;
      float s = acc[i];
#pragma unroll
      for (int k = 0; k < 64; ++k) s = fmaf(w[k], xm[k], s);
      acc[i] = s;
    }
  }
  // RMSNorm row factors 1 / rms(x_m).
  if (a.ssq)
    for (int m = warp; m < M; m += kGemmThreads / 32) {
      float sq = (lane < a.nssq ? a.ssq[lane * kRows + m] : 0.f) + (lane + 32 < a.nssq ? a.ssq[(lane + 32) * kRows + m] : 0.f);
      sq = warp_sum(sq);
      if (lane == 0) s_rinv[m] = 1.0f / sqrtf(sq * a.inv_k + a.eps);
    }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kF32Tok; ++i) {
    const int m = par + 2 * i;
    if (m >= M) break;
    ys[m * kBlockRows + r] = a.ssq ? acc[i] * s_rinv[m] : acc[i];
  }
  __syncthreads();
  const int G = (M + kGroupRows - 1) / kGroupRows;
  for (int m0 = 0; m0 < M; m0 += kGroupRows) {
    const int Mg = min(kGroupRows, M - m0);
    float* yg = ys + m0 * kBlockRows;
    EpiPre<4> pre;
    epi_prefetch<4, EPI, true>(a, rb, m0, Mg, pre, s_pos + m0);
    if (EPI == EPI_RESID) epi_resid<4>(a, yg, rb, m0, Mg, T4, pre);
    else if (EPI == EPI_QKV) epi_qkv<4>(a, yg, rb, m0, Mg, pre, s_pos + m0);
    else if (EPI == EPI_SWIGLU) epi_swiglu(a, yg, rb, m0, Mg, T4);
    else if (EPI == EPI_ARGMAX) epi_argmax(a, yg, rb, m0, Mg, a.nblocks * G, &s_flag);
    else epi_store(a, yg, rb, m0, Mg);
  }
}

static int f32_smem_bytes() { return (kRows * kBlockRows + kRows * 64) * 4; }

template <int EPI>
static cudaError_t launch_f32_t(const GemmArgs& a, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nblocks);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = f32_smem_bytes();
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_gemm_f32<EPI>, a);
}

cudaError_t launch_gemm_f32(const GemmArgs& a, int epi, cudaStream_t st, bool pdl) {
  if (a.rs.M < 1 || a.rs.M > kRows) return cudaErrorInvalidValue;
  switch (epi) {
    case EPI_QKV: return launch_f32_t<EPI_QKV>(a, st, pdl);
    case EPI_RESID: return launch_f32_t<EPI_RESID>(a, st, pdl);
    case EPI_SWIGLU: return launch_f32_t<EPI_SWIGLU>(a, st, pdl);
    case EPI_ARGMAX: return launch_f32_t<EPI_ARGMAX>(a, st, pdl);
    case EPI_STORE: return launch_f32_t<EPI_STORE>(a, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t f32_init() {
  const void* fns[] = {reinterpret_cast<const void*>(k_gemm_f32<EPI_QKV>),
                       reinterpret_cast<const void*>(k_gemm_f32<EPI_RESID>),
                       reinterpret_cast<const void*>(k_gemm_f32<EPI_SWIGLU>),
                       reinterpret_cast<const void*>(k_gemm_f32<EPI_ARGMAX>),
                       reinterpret_cast<const void*>(k_gemm_f32<EPI_STORE>)};
  for (const void* f : fns) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, f32_smem_bytes());
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace sf
