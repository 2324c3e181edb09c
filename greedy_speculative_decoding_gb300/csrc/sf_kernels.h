// Internal launch interface between the engine (host) and the kernels.
#pragma once

#include "sf_common.cuh"

namespace sf {

enum Epi { EPI_QKV = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_ARGMAX = 3, EPI_STORE = 4 };

// Skinny GEMM y[m][n] = sum_k a[m][k] * W[n][k] over up to SF_MAX_ROWS token
// rows (16 per CTA; more run as 16-row groups), with a fused prologue
// (optional RMSNorm of the fp32 input) and one of five epilogues. Weights are bf16 row-major, or NF4 (packed codes + fp16
// block scales) when nf4 != 0.
struct GemmArgs {
  CUtensorMap tm[3];          // per segment: 2-D map {K, rows}, box {64, 16}, 128-byte swizzle
                              // (NF4: codes {K/2 bytes, rows}, box {128, 16}, 128-byte swizzle)
  CUtensorMap tms[3];         // NF4 block scales per segment: {K/64, rows}, box {8, 16}
  const void* w[3];           // row segments (QKV: q, k, v; SWIGLU: gate, up)
  const void* bias[3];        // bf16, or fp32 when wf32
  int seg_end[3];             // cumulative row ends of the segments
  int ld[3];                  // row stride in elements (bf16) / codes (NF4)
  int nseg;
  int nf4;
  int N, K;                   // output rows (SWIGLU: ffn features), reduction length
  int nblocks, nsplit, cps;   // row blocks, K splits, chunks per split
  int stages;                 // weight tiles in flight per warp (2..kMaxStages)
  int push;                   // cluster split: ranks push their tiles into rank 0 (set by launch_gemm)
  int stage_b;                // B operand copied into shared memory first (set by launch_gemm)
  int cluster;                // 1: the splits of a row block form one thread-block
                              // cluster and are summed through distributed shared
                              // memory; 0: through `part` in global memory
  // Input activations in fragment order (frag_index, T = ceil(M / 4)). For
  // the input of an RMSNorm they hold x * gain and ssq is set: the epilogue
  // scales row m by 1 / rms(x_m), computed from the partial sums of squares.
  const uint4* in;
  const float* ssq;           // [nssq][kRows] partial sums of squares of x, or null
  int nssq;
  float eps, inv_k;
  // Fragment-ordered copy of the epilogue's result for the next GEMM: RESID
  // writes x * frag_gain (the next RMSNorm's input), SWIGLU the activation.
  bf16* frag_out;
  const void* frag_gain;      // bf16, or fp32 when wf32
  int frag_umma;              // frag_out in the tensor-core operand order (umma_index) instead of fragment order
  // split-K scratch without clusters: partial tiles [row block x row group][split][16][128]
  // and one arrival counter per (row block, row group)
  float* part;
  int* counter;
  // epilogue outputs
  float* out;                 // QKV: q [M][q_dim]; RESID: x [M][H]; SWIGLU: act [M][F]; STORE: y [M][N]
  int out_ld;
  float* ssq_out;             // RESID: [nblocks][kRows]
  int q_dim, kv_dim, hd, nkv, s_max;
  bf16* kc;                   // this layer's key cache [B][nkv][s_max][hd]
  bf16* vc;
  const float2* rope;         // [s_max][hd/2] (cos, sin)
  unsigned long long* keys;   // ARGMAX: [kRows] packed (value, index)
  int* done;                  // ARGMAX: finished-block counter
  int* tok_out;               // ARGMAX: token of row m -> tok_out[b*tok_stride + tok_off + j - tok_skip]
  int tok_stride, tok_skip, tok_off;   // rows with j < tok_skip produce nothing
  float* logits;              // ARGMAX: optional fp32 rows, row (b*lg_stride + lg_off + j - tok_skip)
  int lg_stride, lg_off;
  int* err;                   // status word (kErr* bits), or null
  int wf32;                   // gains and biases are fp32 (SF_WDTYPE_F32 models)
  int expire_first_wait;      // test hook: the first weight-tile wait reports an expiry
  RowSet rs;
};

// Tensor map of a bf16 weight matrix [rows, K] with row stride ld elements,
// in the layout the GEMM's TMA ring expects: boxes of 64 k x box_rows rows
// with 128-byte swizzle (16 rows: one warp's tile of the mma.sync GEMM; 64
// rows: half the 128-row tile of the tcgen05 GEMM).
cudaError_t make_weight_map(CUtensorMap* map, const void* w, int rows, int K, int ld, int box_rows = 16);
// NF4: codes [rows, K/2] bytes and fp16 block scales [rows, nf4_scale_ld(K)].
int nf4_scale_ld(int K);
cudaError_t make_nf4_maps(CUtensorMap* codes_map, CUtensorMap* scale_map, const void* codes, const void* scales,
                          int rows, int K, int box_rows = 16);
cudaError_t set_nf4_levels(const float levels[16]);

constexpr int kMaxClusterSplit = 16;  // cluster size (above 8 is non-portable; allowed per kernel)
constexpr int kMaxStages = 9;         // deepest bf16 weight ring (beside 16 token rows and their operands)
constexpr int kMaxStagesNF4 = 6;      // NF4 stages also carry their block scales (and a 32 KB table)

// fp32 rows x [M][ld] (features 0..K-1) -> fragment order, zero past K and
// past M within the last token tile (the input of sf_linear).
cudaError_t launch_to_frag(const float* x, int M, int K, int ld, bf16* out, cudaStream_t st);

// Ring depth for a plan. A grid of at most one CTA per SM gets rings of up
// to five stages (under 114 KB of shared memory), so that one CTA of this
// kernel and one of the next fit on an SM together: the next kernel's CTAs
// start early and stream their weights while this one finishes. Larger
// grids run two CTAs per SM with four stages. An NF4 stage holds four chunks.
inline int pick_stages(int ctas, int cps, int num_sms, bool nf4 = false) {
  const int need = nf4 ? (cps + 3) / 4 : cps;
  if (ctas <= num_sms) return need < 2 ? 2 : (need > 5 ? 5 : need);
  return kStages;
}

// A CTA with at least two chunks whose B operand (all its chunks, all token
// tiles) fits in kMaxStagedB bytes copies it into shared memory once after
// its wait instead of loading it from global memory chunk by chunk.
constexpr int kMaxStagedB = 24 * 1024;
__host__ __device__ inline int staged_b_bytes(int T, int cps) {
  return (cps >= 2 && cps * T * 1024 <= kMaxStagedB) ? cps * T * 1024 : 0;
}
// A cluster split whose ranks' partial tiles for rank 0 fit in kMaxPushBytes
// pushes them there with asynchronous remote stores (one hop, no barrier
// round trip); larger ones are pulled by rank 0 after a cluster barrier.
constexpr int kMaxPushBytes = 32 * 1024;
constexpr int kHalfSmBytes = 112 * 1024;   // dynamic shared memory that still lets two CTAs share an SM
__host__ __device__ inline int push_bytes(int nsplit, int M) { return (nsplit - 1) * M * kBlockRows * 4; }
int gemm_smem_bytes(int M, int stages, bool nf4, int cps, int push = 0);
int gemm_max_clusters(int csize, int M, int stages, int cps);
cudaError_t gemm_init();
cudaError_t launch_gemm(const GemmArgs& a, int epi, cudaStream_t st, bool pdl);
// The same projections on the tcgen05 tensor cores for launches of 17 to
// SF_MAX_ROWS token rows (k_umma.cu): one CTA per (128 weight rows, K slice)
// covers every token row; the input is in the tensor-core operand order
// (umma_index), the weight maps have 64-row boxes, the K slices of a row
// block are one cluster (at most 8) or use `part` / `counter`.
cudaError_t launch_umma(const GemmArgs& a, int epi, cudaStream_t st, bool pdl);
int umma_min_rows();
int umma_min_rows_nf4();
cudaError_t umma_init();
int umma_smem_bytes(int M, int stages, bool nf4);
int umma_stages(int M, bool nf4);
int umma_max_clusters(int csize, int M, int stages, bool nf4);
cudaError_t set_umma_nf4_levels(const float levels[16]);
// The LM head with its argmax as a persistent kernel (one K slice, at most
// two CTAs per SM walking the row blocks); same arguments as EPI_ARGMAX.
cudaError_t launch_lmhead(const GemmArgs& a, int num_sms, cudaStream_t st, bool pdl);
// The projections of SF_WDTYPE_F32 models (k_f32.cu): fp32 weights (plain
// pointers, row stride ld), one CTA per 128 output rows, any row count up to
// SF_MAX_ROWS, inputs in fragment order, the same epilogues.
cudaError_t launch_gemm_f32(const GemmArgs& a, int epi, cudaStream_t st, bool pdl);
cudaError_t f32_init();

struct EmbedArgs {
  const void* E;   // bf16, or fp32 when f32
  int ld, H, vocab;
  int* err;
  float* x;      // [M][H]
  float* ssq;    // [H/128][kRows]
  bf16* frag;    // x * gain in fragment order (the first RMSNorm's input)
  const void* gain;
  int f32;       // embedding and gain in fp32
  int umma;      // frag in the tensor-core operand order instead
  RowSet rs;
};
cudaError_t launch_embed(const EmbedArgs& a, cudaStream_t st, bool pdl);

struct AttnArgs {
  // The model's whole KV cache as a 2-D tensor of head_dim-wide bf16 rows
  // (box 64 x 64, 128-byte swizzle): the keys of (sequence b, KV head h,
  // slot p) of this layer are row kv_row0 + b * kv_brows + h * s_max + p, the
  // values kv_vrows rows further.
  CUtensorMap kvmap;
  CUtensorMap kvmap8;      // the same with 8-slot boxes: a sequence's partly filled last chunk
  const bf16* kc;          // this layer's keys [B][nkv][s_max][hd] (the one-chunk copy kernel)
  const bf16* vc;          // and values
  int box8;                // 1: load a partly filled last chunk in 8-slot boxes
  int kv_row0, kv_brows, kv_vrows;
  int R;                   // cache chunks per work item (one partial result per R chunks)
  int TG;                  // 16-query tiles per work item (1..4)
  int stages;              // key/value chunks in flight per CTA (1 or 2)
  const float* q;          // [M][nq*hd], RoPE applied
  float* part;             // [M*nq][n_kv_chunks][hd + 2]: partial results per R-chunk range
  bf16* out;               // attention output [M][nq*hd] in fragment order
  int umma;                // out in the tensor-core operand order instead
  int nq, nkv, hd, s_max, B, n_kv_chunks;
  float scale;
  int* err;
  int merge_trace_id;      // timeline slot of the merge kernel
  RowSet rs;
};
cudaError_t launch_attention(const AttnArgs& a, int num_sms, cudaStream_t st, bool pdl);
// Tensor map of a KV cache [rows][hd] bf16 (rows = layers * 2 * batch * n_kv_heads * s_max).
cudaError_t make_kv_map(CUtensorMap* map, const void* kv, long rows, int hd, int box_rows = 64);
// Shared-memory limits and carve-out of the attention kernels (current device).
cudaError_t attn_init();

cudaError_t launch_rope_table(float2* table, int s_max, int hd, float theta, cudaStream_t st);

// Engine state on the device (one sequence per b).
struct SpecState {
  int* len_t;       // [B] target cache length = committed - 1
  int* len_d;       // [B] draft cache slots known valid (committed - 2)
  int* vtok;        // [B][K+1] verify rows: pending, d_1..d_K
  int* ttok;        // [B][K+1] target argmax per verify row
  int* dtok0;       // [B][2] first draft step rows: the last two committed tokens
  int* nprop;       // [B] real guesses this round
  int* hist;        // [B][s_max] committed tokens
  int* ncommit;     // [B] tokens committed by the last round
  int* nacc;        // [B] accepted guesses of the last round
  int* commit;      // [B][K+1] tokens committed by the last round
  int* total;       // [B] tokens generated since prefill
  int* acc_hist;    // [B][K+1] accept-length histogram
  int* prompt_len;  // [B]
  int* err;
  int* loop_target; // device-resident loop: new tokens per sequence to reach
  int* rounds;      // device-resident loop: rounds run by the current sf_generate
  int* clen;        // [B][K] multi-candidate draft: tokens of each candidate guess (0: none)
  int* tree_c;      // [B] multi-candidate draft: the candidate the last round took
  int B, K, s_max;
};

// The persistent decode forward (k_decode.cu): bf16 weights of one layer.
struct DecLayer {
  const bf16 *ln1, *wq, *wk, *wv, *bq, *bk, *bv, *wo, *ln2, *wg, *wu, *wd;
};
struct DecArgs {
  const DecLayer* layers;   // device array [L]
  int L, H, nq, nkv, hd, F, vocab;
  const bf16* embed;
  int embed_ld;
  const bf16* norm;         // final RMSNorm gain
  float eps, scale;
  const float2* rope;       // [s_max][hd / 2]
  bf16* kv;                 // the model's cache [L][2][B][nkv][s_max][hd]
  int B, s_max;
  RowSet rs;                // M <= 4 rows
  int R;                    // cache chunks per attention range
  int n_ranges;             // range stride of `part` (>= ranges of the longest row)
  float* x;                 // [M][H] residual stream
  float* q;                 // [M][nq * hd]
  float* part;              // [M][nq][n_ranges][hd + 2] attention partials
  float* h;                 // [M][F] SwiGLU output
  bf16* frag;               // LM-head input, fragment order
  float* ssq;               // [H / 128][kRows] sums of squares for the LM head
  unsigned* bar;            // grid barrier {count, generation}
  unsigned* cnt;            // [B][nkv] attention items finished (zero between launches)
  int* err;
  int expire_first_wait;    // test hook: the first barrier reports an expired wait
};
int decode_smem_bytes(int MR, int H, int QD, int F, int hd, int group, int rps, int n_ranges);
cudaError_t decode_init(int max_smem);
cudaError_t launch_decode(const DecArgs& a, int num_sms, cudaStream_t st);

// Record a message for sf_last_error() and return `s`.
sf_status set_error(sf_status s, const char* fmt, ...);

cudaError_t launch_accept(const SpecState& s, int mode, cudaStream_t st, bool pdl);
cudaError_t launch_ngram(const SpecState& s, int max_guess, int min_n, int max_n, int* d_prop,
                         int* d_count, cudaStream_t st, bool pdl);
cudaError_t launch_reset(const SpecState& s, cudaStream_t st);
// Multi-candidate prompt lookup: up to n_cand guesses of up to g tokens
// (g * n_cand <= K) into the verify rows; its acceptance over the candidates
// (the longest accepted prefix wins, the lowest candidate on ties); and the
// move of the winner's cache entries down to the committed slots of every
// layer (kv: one model's cache, [layers][2][B][nkv][s_max][hd] bf16).
cudaError_t launch_ngram_tree(const SpecState& s, int n_cand, int g, int min_n, int max_n, int* d_prop,
                              int* d_len, cudaStream_t st, bool pdl);
cudaError_t launch_accept_tree(const SpecState& s, int n_cand, int g, cudaStream_t st, bool pdl);
cudaError_t launch_tree_compact(const SpecState& s, bf16* kv, int layers, int nkv, int hd, int g, cudaStream_t st,
                                bool pdl);
// Device-resident round loop: set the target and clear the round count
// (before the loop graph), and the control kernel at the end of every round
// that decides whether the loop runs another round.
cudaError_t launch_loop_init(const SpecState& s, int n_new, cudaStream_t st);
cudaError_t launch_loop_ctl(const SpecState& s, cudaGraphConditionalHandle h, cudaStream_t st);
cudaError_t launch_copy_draft(const SpecState& s, int* d_draft, cudaStream_t st);
void nf4_levels(double out[16]);
cudaError_t launch_nf4_quantize(const bf16* w, int rows, int cols, int ld, uint8_t* packed,
                                __half* scales, int scale_ld, cudaStream_t st);

}  // namespace sf
