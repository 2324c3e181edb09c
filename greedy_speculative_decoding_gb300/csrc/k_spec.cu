// Integer kernels of the speculative round: accept + in-place rollback,
// prompt-lookup (n-gram) drafting with one guess or several (with their
// acceptance and cache compaction), state reset; and the NF4 codebook and
// quantiser used to prepare 4-bit weights.
#include <cmath>

#include "sf_kernels.h"

namespace sf {

namespace {
cudaLaunchAttribute pdl_attr() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}
}  // namespace

// ---------------------------------------------------------------- accept
// One warp per sequence. Lane j compares guess d_{j+1} with the target's
// choice t_j; the first mismatch (or the number of real guesses) is the
// accepted length n. d_1..d_n and t_n are committed; the target cache keeps
// committed - 1 entries and the draft cache committed - 2 (its next first
// step rewrites the last two slots). Nothing in the caches moves.
__global__ void k_accept(const __grid_constant__ SpecState s, int ngram) {
  pdl_wait();
  pdl_launch_next();
  const int b = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (b >= s.B) return;
  const int K1 = s.K + 1;
  const int* vt = s.vtok + b * K1;      // pending, d_1..d_K
  const int* tt = s.ttok + b * K1;      // t_0..t_K
  const int limit = ngram ? min(s.nprop[b], s.K) : s.K;
  const bool stop = lane >= limit || vt[1 + lane] != tt[lane];
  const int n = __ffs(__ballot_sync(0xffffffffu, stop)) - 1;   // lane `limit` always stops
  const int C = s.len_t[b] + 1;                                  // committed before this round
  int tok = 0;
  if (lane <= n) tok = lane < n ? vt[1 + lane] : tt[n];
  const int before_last = n > 0 ? vt[n] : vt[0];
  __syncwarp();
  if (lane <= n) {
    s.commit[b * K1 + lane] = tok;
    if (C + lane < s.s_max) s.hist[(size_t)b * s.s_max + C + lane] = tok;
  }
  if (lane == 0) {
    const int Cn = C + n + 1;
    s.len_t[b] = Cn - 1;
    s.len_d[b] = Cn - 2;
    s.ncommit[b] = n + 1;
    s.nacc[b] = n;
    s.total[b] += n + 1;
    s.acc_hist[b * K1 + n] += 1;
    s.dtok0[2 * b] = before_last;
    s.dtok0[2 * b + 1] = tt[n];
    s.vtok[b * K1] = tt[n];
    if (Cn + s.K + 1 > s.s_max) atomicOr(s.err, kErrCapacity);
  }
}

cudaError_t launch_accept(const SpecState& s, int mode, cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attr = pdl_attr();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32 * s.B);
  cfg.stream = st;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_accept, s, mode != SF_DRAFT_NEURAL ? 1 : 0);
}

// ---------------------------------------------------------------- n-gram
// One CTA per sequence over its committed tokens ctx[0..C). For n = max_n
// down to min_n: the largest j < C - n with ctx[j..j+n) == ctx[C-n..C) (the
// rightmost earlier occurrence, which may overlap the suffix); the guess is
// ctx[j+n .. min(j+n+max_guess, C)).
__global__ void k_ngram(const __grid_constant__ SpecState s, int max_guess, int min_n, int max_n,
                        int* d_prop, int* d_count) {
  pdl_wait();
  pdl_launch_next();
  __shared__ int best;
  const int b = blockIdx.x;
  const int C = s.len_t[b] + 1;
  const int* ctx = s.hist + (size_t)b * s.s_max;
  int found_j = -1, found_n = 0;
  for (int n = max_n; n >= min_n; --n) {
    if (n > C - 1) continue;
    if (threadIdx.x == 0) best = -1;
    __syncthreads();
    int mine = -1;
    for (int j = C - n - 1 - (int)threadIdx.x; j >= 0; j -= blockDim.x) {
      bool eq = true;
      for (int i = 0; i < n && eq; ++i) eq = ctx[j + i] == ctx[C - n + i];
      if (eq) {
        mine = j;
        break;   // j only decreases for this thread
      }
    }
    if (mine >= 0) atomicMax(&best, mine);
    __syncthreads();
    const int bj = best;
    __syncthreads();
    if (bj >= 0) {
      found_j = bj;
      found_n = n;
      break;
    }
  }
  if (threadIdx.x == 0) {
    int cnt = 0;
    if (found_j >= 0) cnt = min(max_guess, C - (found_j + found_n));
    const int K1 = s.K + 1;
    for (int i = 0; i < s.K; ++i) {
      const int tok = i < cnt ? ctx[found_j + found_n + i] : 0;
      s.vtok[b * K1 + 1 + i] = tok;
      if (d_prop && i < max_guess) d_prop[b * max_guess + i] = tok;
    }
    s.nprop[b] = cnt;
    if (d_count) d_count[b] = cnt;
  }
}

cudaError_t launch_ngram(const SpecState& s, int max_guess, int min_n, int max_n, int* d_prop,
                         int* d_count, cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attr = pdl_attr();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(s.B);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_ngram, s, max_guess, min_n, max_n, d_prop, d_count);
}

// ---------------------------------------------------------------- several guesses
// Multi-candidate prompt lookup, one CTA per sequence. The earlier
// occurrences of the context's last n tokens are visited in k_ngram's order
// (n from max_n down to min_n; for each n the rightmost start first); each
// gives the up to g tokens that followed it, cut at the end of the context,
// and is kept unless it equals a guess already kept; at most n_cand. Every
// step tests 256 starts at once; warp 0 walks that step's matches in visit
// order and keeps the new ones. Candidate c's guess fills verify rows
// 1 + c * g .. c * g + g (unused rows: token 0).
constexpr int kTreeThreads = 256;

__global__ void __launch_bounds__(kTreeThreads) k_ngram_tree(const __grid_constant__ SpecState s, int n_cand,
                                                             int g, int min_n, int max_n, int* d_prop,
                                                             int* d_len) {
  pdl_wait();
  pdl_launch_next();
  __shared__ int kept_at[32], kept_len[32];
  __shared__ unsigned ballot[kTreeThreads / 32];
  __shared__ int nkept;
  const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = s.len_t[b] + 1;
  const int* ctx = s.hist + (size_t)b * s.s_max;
  if (tid == 0) nkept = 0;
  __syncthreads();
  for (int n = max_n; n >= min_n; --n) {
    if (n > C - 1) continue;
    for (int top = C - n - 1; top >= 0 && nkept < n_cand; top -= kTreeThreads) {
      const int j = top - tid;
      bool eq = j >= 0;
      for (int i = 0; i < n && eq; ++i) eq = ctx[j + i] == ctx[C - n + i];
      const unsigned bal = __ballot_sync(0xffffffffu, eq);
      if (lane == 0) ballot[warp] = bal;
      if (!__syncthreads_or(eq)) continue;
      if (warp == 0) {
        // Lower thread = larger start = earlier in visit order.
        for (int w = 0; w < kTreeThreads / 32 && nkept < n_cand; ++w) {
          unsigned m = ballot[w];
          while (m && nkept < n_cand) {
            const int t = __ffs(m) - 1;
            m &= m - 1;
            const int at = top - (32 * w + t) + n, len = min(g, C - at);
            // Lane k < nkept compares this guess with kept guess k.
            bool dup = false;
            if (lane < nkept && kept_len[lane] == len) {
              dup = true;
              for (int i = 0; i < len && dup; ++i) dup = ctx[kept_at[lane] + i] == ctx[at + i];
            }
            if (!__any_sync(0xffffffffu, dup)) {
              if (lane == 0) {
                kept_at[nkept] = at;
                kept_len[nkept] = len;
                nkept = nkept + 1;
              }
            }
            __syncwarp();
          }
        }
      }
      __syncthreads();
    }
  }
  const int K1 = s.K + 1;
  for (int r = tid; r < s.K; r += kTreeThreads) {
    const int c = r / g, i = r - c * g;
    const int tok = (c < nkept && i < kept_len[c]) ? ctx[kept_at[c] + i] : 0;
    s.vtok[b * K1 + 1 + r] = tok;
    if (d_prop && c < n_cand) d_prop[(b * n_cand + c) * g + i] = tok;
  }
  for (int c = tid; c < s.K; c += kTreeThreads) {
    const int len = c < nkept ? kept_len[c] : 0;
    s.clen[b * s.K + c] = len;
    if (d_len && c < n_cand) d_len[b * n_cand + c] = len;
  }
  if (tid == 0) s.nprop[b] = nkept;
}

cudaError_t launch_ngram_tree(const SpecState& s, int n_cand, int g, int min_n, int max_n, int* d_prop,
                              int* d_len, cudaStream_t st, bool pdl) {
  if (n_cand < 1 || g < 1 || n_cand * g > s.K || n_cand > 32) return cudaErrorInvalidValue;
  cudaLaunchAttribute attr = pdl_attr();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(s.B);
  cfg.blockDim = dim3(kTreeThreads);
  cfg.stream = st;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_ngram_tree, s, n_cand, g, min_n, max_n, d_prop, d_len);
}

// Acceptance over the candidates, one warp per sequence. Lane c counts the
// leading tokens of candidate c that equal the target's choices along that
// candidate's own rows: the choice after the pending token is row 0's, the
// choice after guess tokens 0..i-1 of candidate c is row c * g + i's. The
// longest count wins, the lowest candidate on ties; its accepted tokens and
// the choice after them are committed, as in k_accept.
__global__ void k_accept_tree(const __grid_constant__ SpecState s, int n_cand, int g) {
  pdl_wait();
  pdl_launch_next();
  const int b = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (b >= s.B) return;
  const int K1 = s.K + 1;
  const int* vt = s.vtok + b * K1;
  const int* tt = s.ttok + b * K1;
  int key = -1;
  if (lane < n_cand) {
    const int len = s.clen[b * s.K + lane];
    int n = 0;
    while (n < len && vt[1 + lane * g + n] == tt[n == 0 ? 0 : lane * g + n]) ++n;
    key = n * 32 + (31 - lane);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, o));
  const int n = key >> 5, c = 31 - (key & 31);
  const int C = s.len_t[b] + 1;
  const int last = tt[n == 0 ? 0 : c * g + n];
  int tok = 0;
  if (lane <= n) tok = lane < n ? vt[1 + c * g + lane] : last;
  const int before_last = n > 0 ? vt[c * g + n] : vt[0];
  __syncwarp();
  if (lane <= n) {
    s.commit[b * K1 + lane] = tok;
    if (C + lane < s.s_max) s.hist[(size_t)b * s.s_max + C + lane] = tok;
  }
  if (lane == 0) {
    const int Cn = C + n + 1;
    s.len_t[b] = Cn - 1;
    s.len_d[b] = Cn - 2;
    s.ncommit[b] = n + 1;
    s.nacc[b] = n;
    s.tree_c[b] = c;
    s.total[b] += n + 1;
    s.acc_hist[b * K1 + n] += 1;
    s.dtok0[2 * b] = before_last;
    s.dtok0[2 * b + 1] = last;
    s.vtok[b * K1] = last;
    if (Cn + s.K + 1 > s.s_max) atomicOr(s.err, kErrCapacity);
  }
}

cudaError_t launch_accept_tree(const SpecState& s, int n_cand, int g, cudaStream_t st, bool pdl) {
  if (n_cand < 1 || g < 1 || n_cand * g > s.K || n_cand > 32) return cudaErrorInvalidValue;
  cudaLaunchAttribute attr = pdl_attr();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32 * s.B);
  cfg.stream = st;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_accept_tree, s, n_cand, g);
}

// The verify pass wrote candidate c's guess i into slot C + c * g + i; the
// accepted ones belong in slots C + i. One CTA per (layer, sequence) moves
// the n accepted keys and values of every KV head, 16 bytes per thread step.
// Source and destination never overlap (n <= g <= c * g for c >= 1).
__global__ void k_tree_compact(const __grid_constant__ SpecState s, bf16* kv, int nkv, int hd, int g) {
  pdl_wait();
  pdl_launch_next();
  const int l = blockIdx.x, b = blockIdx.y;
  const int c = s.tree_c[b], n = s.nacc[b];
  if (c == 0 || n == 0) return;
  const int C = s.len_t[b] - n;
  const int units = hd / 8;   // 16-byte pieces of one cache row
  const int per_head = n * units;
  for (int i = threadIdx.x; i < 2 * nkv * per_head; i += blockDim.x) {
    const int kvsel = i / (nkv * per_head);
    const int rest = i - kvsel * nkv * per_head;
    const int h = rest / per_head, rr = rest - h * per_head;
    const int row = rr / units, u = rr - row * units;
    bf16* base = kv + ((((size_t)l * 2 + kvsel) * s.B + b) * nkv + h) * (size_t)s.s_max * hd;
    const uint4 v = *reinterpret_cast<const uint4*>(base + (size_t)(C + c * g + row) * hd + 8 * u);
    *reinterpret_cast<uint4*>(base + (size_t)(C + row) * hd + 8 * u) = v;
  }
}

cudaError_t launch_tree_compact(const SpecState& s, bf16* kv, int layers, int nkv, int hd, int g, cudaStream_t st,
                                bool pdl) {
  if (hd % 8 || g < 1) return cudaErrorInvalidValue;
  cudaLaunchAttribute attr = pdl_attr();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(layers, s.B);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_tree_compact, s, kv, nkv, hd, g);
}

// ---------------------------------------------------------------- device loop
// sf_generate as one graph launch: a WHILE conditional node whose body is one
// round followed by k_loop_ctl. The control kernel counts the round and lets
// the loop run again while some sequence has fewer than the target number of
// new tokens, every sequence has room for two more rounds (so acceptance
// never raises the capacity flag), no error bit is set, and fewer rounds than
// the target have run (each round commits at least one token per sequence,
// so that bound never stops a loop that still has work).
__global__ void k_loop_init(const __grid_constant__ SpecState s, int n_new) {
  *s.loop_target = n_new;
  *s.rounds = 0;
}

__global__ void k_loop_ctl(const __grid_constant__ SpecState s, cudaGraphConditionalHandle h) {
  const int r = *s.rounds + 1;
  *s.rounds = r;
  const int target = *s.loop_target;
  bool need = false, room = true;
  for (int b = 0; b < s.B; ++b) {
    need = need || s.total[b] < target;
    room = room && s.len_t[b] + 1 + 2 * (s.K + 1) <= s.s_max;
  }
  cudaGraphSetConditional(h, (need && room && *s.err == 0 && r < target) ? 1u : 0u);
}

cudaError_t launch_loop_init(const SpecState& s, int n_new, cudaStream_t st) {
  k_loop_init<<<1, 1, 0, st>>>(s, n_new);
  return cudaGetLastError();
}

cudaError_t launch_loop_ctl(const SpecState& s, cudaGraphConditionalHandle h, cudaStream_t st) {
  k_loop_ctl<<<1, 1, 0, st>>>(s, h);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- reset
// Back to "prompt prefilled": caches hold prompt[0..P-1), prompt[P-1] pending.
__global__ void k_reset(const __grid_constant__ SpecState s) {
  const int b = threadIdx.x;
  if (b >= s.B) return;
  const int P = s.prompt_len[b];
  const int* h = s.hist + (size_t)b * s.s_max;
  s.len_t[b] = P - 1;
  s.len_d[b] = P - 2;
  s.vtok[b * (s.K + 1)] = h[P - 1];
  s.dtok0[2 * b] = h[P - 2];
  s.dtok0[2 * b + 1] = h[P - 1];
  s.total[b] = 0;
  s.ncommit[b] = 0;
  s.nacc[b] = 0;
  s.nprop[b] = 0;
  for (int i = 0; i <= s.K; ++i) s.acc_hist[b * (s.K + 1) + i] = 0;
}

cudaError_t launch_reset(const SpecState& s, cudaStream_t st) {
  k_reset<<<1, 32, 0, st>>>(s);
  return cudaGetLastError();
}

__global__ void k_copy_draft(const __grid_constant__ SpecState s, int* d_draft) {
  const int i = threadIdx.x;
  if (i < s.B * s.K) {
    const int b = i / s.K, j = i - b * s.K;
    d_draft[i] = s.vtok[b * (s.K + 1) + 1 + j];
  }
}

cudaError_t launch_copy_draft(const SpecState& s, int* d_draft, cudaStream_t st) {
  k_copy_draft<<<1, 256, 0, st>>>(s, d_draft);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- NF4
// NormalFloat levels (Dettmers et al., "QLoRA", 2023, section 3): normal
// quantiles on evenly spaced probabilities from 1/2 to `edge`, 8 on the
// positive side and 7 on the negative side, plus an exact zero, scaled to
// [-1, 1]. `edge` is the midpoint of the outermost probabilities of 16- and
// 15-point grids, which keeps the end levels finite. The quantile x of
// probability p solves Phi(x) = p with Phi(x) = erfc(-x / sqrt 2) / 2; it is
// found by Newton's method from x = 0 (Phi is concave on x >= 0, so every
// tangent lies above it and the iterates rise monotonically to the root).
static double normal_quantile_upper(double p) {
  const double inv_sqrt2 = 0.70710678118654752440;
  const double inv_sqrt2pi = 0.39894228040143267794;
  double x = 0.0;
  for (int it = 0; it < 100; ++it) {
    const double f = 0.5 * std::erfc(-x * inv_sqrt2) - p;
    const double dx = f / (inv_sqrt2pi * std::exp(-0.5 * x * x));
    x -= dx;
    if (std::fabs(dx) < 1e-17) break;
  }
  return x;
}

void nf4_levels(double out[16]) {
  const double edge = 0.5 * ((1.0 - 1.0 / 32.0) + (1.0 - 1.0 / 30.0));
  const double top = normal_quantile_upper(edge);
  for (int i = 0; i < 7; ++i) out[i] = -normal_quantile_upper(edge - (edge - 0.5) * i / 7.0) / top;
  out[7] = 0.0;
  for (int i = 0; i < 8; ++i) out[8 + i] = normal_quantile_upper(0.5 + (edge - 0.5) * (i + 1) / 8.0) / top;
  out[0] = -1.0;
  out[15] = 1.0;
}

// One warp per 64-element block: scale = fp16(max |w|); code = number of fp32
// midpoints of adjacent fp32 levels strictly below w / scale (ties -> lower
// code); two codes per byte, element 2i in the low nibble.
__constant__ float c_nf4_mid[15];

__global__ void k_nf4_quantize(const bf16* w, int rows, int cols, int ld, uint8_t* packed,
                               __half* scales, int scale_ld) {
  const long warp = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int nblk = cols / 64;
  if (warp >= (long)rows * nblk) return;
  const int r = (int)(warp / nblk), blk = (int)(warp - (long)r * nblk);
  const bf16* src = w + (size_t)r * ld + blk * 64 + 2 * lane;
  const float a = __bfloat162float(src[0]), b = __bfloat162float(src[1]);
  const float amax = warp_max(fmaxf(fabsf(a), fabsf(b)));
  const __half sh = __float2half_rn(amax);
  const float sc = __half2float(sh);
  int ca = 7, cb = 7;
  if (sc > 0.f) {
    const float xa = __fdiv_rn(a, sc), xb = __fdiv_rn(b, sc);
    ca = 0;
    cb = 0;
#pragma unroll
    for (int i = 0; i < 15; ++i) {
      ca += xa > c_nf4_mid[i];
      cb += xb > c_nf4_mid[i];
    }
  }
  packed[(size_t)r * (cols / 2) + blk * 32 + lane] = (uint8_t)(ca | (cb << 4));
  if (lane == 0) scales[(size_t)r * scale_ld + blk] = sh;
}

cudaError_t launch_nf4_quantize(const bf16* w, int rows, int cols, int ld, uint8_t* packed,
                                __half* scales, int scale_ld, cudaStream_t st) {
  double lv[16];
  nf4_levels(lv);
  float mids[15];
  for (int i = 0; i < 15; ++i) mids[i] = ((float)lv[i] + (float)lv[i + 1]) * 0.5f;
  cudaError_t e = cudaMemcpyToSymbolAsync(c_nf4_mid, mids, sizeof(mids), 0, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return e;
  const long warps = (long)rows * (cols / 64);
  const int threads = 256;
  const long blocks = (warps * 32 + threads - 1) / threads;
  k_nf4_quantize<<<(unsigned)blocks, threads, 0, st>>>(w, rows, cols, ld, packed, scales, scale_ld);
  return cudaGetLastError();
}

}  // namespace sf
