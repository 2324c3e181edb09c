/*
 * sf.h — C ABI of the GB300 greedy speculative-decoding engine.
 *
 * One speculative round (the hot path) has four parts:
 *   draft    — a small draft model decodes K tokens greedily over its own
 *              static KV cache (sf_draft), or prompt lookup proposes up to K
 *              tokens (sf_ngram_draft);
 *   verify   — the target model runs one causal pass over the pending token
 *              and the K guesses and returns its own greedy choice at every
 *              position (sf_verify);
 *   accept   — the longest prefix of guesses that agrees with the target's
 *              choices is accepted, and the target's choice after it (the
 *              bonus token) is committed as well;
 *   rollback — both KV caches are cut back, in place, to the last committed
 *              position (sf_accept_rollback).
 * sf_step runs all four as one CUDA graph replay.
 *
 * Sources (page title, then section):
 *   "I Got 28 TPS Out of Free Kaggle GPUs. Here's What It Took." —
 *     "Speculative Decoding: The Idea" (draft guesses K tokens, the target
 *     checks them in one pass, agreed tokens are committed);
 *     "CUDA Graphs: What They Are and Why They Helped" (the whole draft
 *     forward, LM head and argmax replayed as one driver call);
 *     "Why It Kept Breaking (and How I Fixed It)" (static preallocated KV
 *     cache, in-place intermediates, explicit position updates, in-place KV
 *     rewind on rejection).
 *   "Qwen3.5-397B on 20 GPUs, through a relay" (Sangama results) —
 *     "Speculative decoding: correct, but slower (for now)" (look-back
 *     guesses of up to 4 tokens from the last 2-4 tokens; the verifier returns
 *     its own choice at every position; output equals normal decoding).
 *
 * Conventions for every call:
 *   - Ownership: the caller allocates and owns every device buffer (weights,
 *     both KV caches, the workspace). They must stay valid until sf_destroy.
 *     The library never allocates device memory; it allocates a little
 *     pinned host memory and one CUDA stream in sf_create.
 *   - Streams: all device work is enqueued on the stream given to sf_create.
 *     Calls that return host results synchronise that stream.
 *   - Errors: every call returns an sf_status and never aborts. On
 *     SF_ERR_ARG, SF_ERR_CAPACITY or SF_ERR_STATE nothing was enqueued and
 *     the engine state is unchanged. sf_last_error() gives a message for the
 *     calling thread's last failure.
 *   - Batch: sequences are independent; per-sequence lengths and accept
 *     lengths are kept on the device.
 *   - Rows per forward (batch * (K + 1)) are limited to SF_MAX_ROWS. Every
 *     forward reads each weight from HBM once: up to 16 bf16 rows on the
 *     weight-streaming mma.sync GEMM (all rows in one pass per CTA), more
 *     rows and every NF4 forward on the tcgen05 GEMM (tensor-memory
 *     accumulators, all token rows as the MMA's N side).
 */
#ifndef SF_H_
#define SF_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SF_API __attribute__((visibility("default")))
#else
#define SF_API
#endif

#define SF_MAX_ROWS 80

typedef struct sf_engine* sf_handle;

typedef enum {
  SF_OK = 0,
  SF_ERR_ARG = 1,          /* invalid argument, null or misaligned pointer */
  SF_ERR_CAPACITY = 2,     /* a round would write past s_max cache slots */
  SF_ERR_CUDA = 3,         /* a CUDA runtime call failed */
  SF_ERR_NONFINITE = 4,    /* a non-finite logit was produced */
  SF_ERR_STATE = 5,        /* call out of order (e.g. verify before draft) */
  SF_ERR_UNSUPPORTED = 6,  /* shape or mode not supported by this build */
  SF_ERR_DEVICE = 7        /* a kernel reported a bounded wait that expired */
} sf_status;

/* Weight types: bf16; NF4 for the 7 linear maps of every layer (embedding,
 * norms, biases and LM head stay bf16); or fp32 for every tensor (the
 * single-precision correctness workload; plain fp32 arithmetic, not a fast path). */
enum { SF_WDTYPE_BF16 = 0, SF_WDTYPE_NF4 = 1, SF_WDTYPE_F32 = 2 };
/* Drafters: the draft model, prompt lookup, none (each round then commits
 * only the target's own next token: plain greedy decoding, the baseline the
 * speculative rounds are measured against), or prompt lookup with several
 * guesses verified side by side in one target pass (sf_tree_draft). */
enum { SF_DRAFT_NEURAL = 0, SF_DRAFT_NGRAM = 1, SF_DRAFT_NONE = 2, SF_DRAFT_TREE = 3 };

/* Decoder shape (Qwen2-style: GQA attention with RoPE, RMSNorm, SwiGLU MLP). */
typedef struct {
  int32_t layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab;
  int32_t tied;       /* 1: the LM head is the embedding matrix */
  int32_t qkv_bias;   /* 1: q, k, v projections carry biases */
  int32_t embed_ld;   /* row stride of the embedding in elements; 0 = hidden */
  float rope_theta;   /* RoPE base */
  float rms_eps;      /* RMSNorm epsilon */
  int32_t wdtype;     /* SF_WDTYPE_BF16, SF_WDTYPE_NF4 or SF_WDTYPE_F32 */
} sf_model_cfg;

/*
 * Weight pointers (device, row-major [out, in], bf16 unless stated; every
 * tensor fp32 with SF_WDTYPE_F32), in this
 * order: embed [vocab, hidden] (row stride embed_ld); per layer: ln1 [hidden],
 * wq [n_heads*head_dim, hidden], wk, wv [n_kv_heads*head_dim, hidden],
 * bq, bk, bv (NULL when qkv_bias == 0), wo [hidden, n_heads*head_dim],
 * ln2 [hidden], wg, wu [ffn, hidden], wd [hidden, ffn]; final norm [hidden];
 * lm_head [vocab, hidden] (omitted when tied).
 * With SF_WDTYPE_NF4 each of wq, wk, wv, wo, wg, wu, wd takes two consecutive
 * slots: packed codes (uint8 [out, in/2], element 2i in the low nibble) then
 * block scales (fp16 [out, ld_s], ld_s = 8 * ceil(in / 512): the in/64 scales
 * of a row padded to a 16-byte row stride), as sf_nf4_quantize writes them;
 * in must be a multiple of 64.
 * Every row must start on a 16-byte boundary.
 * Returns the number of slots, or -1 for an invalid cfg.
 */
SF_API int32_t sf_weight_count(const sf_model_cfg* cfg);

/* Bytes of one KV cache: layout [layers][2 (k, v)][batch][n_kv_heads][s_max][head_dim] bf16. */
SF_API size_t sf_kv_bytes(const sf_model_cfg* cfg, int32_t batch, int32_t s_max);

/* Bytes of device workspace sf_create needs (dft may be NULL: n-gram only);
 * 0 for an invalid configuration. The caller allocates it once: the pages'
 * fix for graph replays is a static, preallocated cache and in-place
 * intermediates ("Why It Kept Breaking (and How I Fixed It)", fixes 1-2). */
SF_API size_t sf_workspace_bytes(const sf_model_cfg* tgt, const sf_model_cfg* dft, int32_t batch,
                          int32_t K, int32_t s_max);

/*
 * Bind caller-owned buffers and build the engine ("Speculative Decoding: The
 * Idea": a small draft model beside the target; for an n-gram-only engine,
 * "Speculative decoding: correct, but slower (for now)" on the Sangama
 * page). kv_d may be NULL when dft
 * is NULL. workspace must hold sf_workspace_bytes(...) bytes, 256-byte
 * aligned. batch: 1..32 independent sequences. K: guesses per round (1..15,
 * batch*(K+1) <= SF_MAX_ROWS).
 * s_max: cache slots per sequence, a multiple of 64.
 * cuda_stream: a cudaStream_t (NULL = legacy default stream).
 * The engine starts with SF_DRAFT_NEURAL when dft is given, else
 * SF_DRAFT_NGRAM (max guess K, n from 4 down to 2).
 */
SF_API sf_status sf_create(const sf_model_cfg* tgt, const void* const* tgt_w,
                    const sf_model_cfg* dft, const void* const* dft_w,
                    int32_t batch, int32_t K, int32_t s_max,
                    void* kv_t, void* kv_d, void* workspace, void* cuda_stream,
                    sf_handle* out);

/*
 * Load prompts and fill both caches (the step before the speculative loop;
 * "Qwen3.5-397B on 20 GPUs", "What made it faster": prompts go through in
 * pieces). h_tokens: host [batch][stride] int32,
 * h_lens: host [batch] prompt lengths (each >= 2 and <= stride; they may
 * differ). After it, each cache holds its prompt except the last token,
 * which is pending. Prompts of one length are filled side by side in chunks
 * of up to SF_MAX_ROWS rows; otherwise each sequence is filled on its own.
 */
SF_API sf_status sf_prefill(sf_handle h, const int32_t* h_tokens, const int32_t* h_lens, int32_t stride);

/*
 * Neural draft ("Speculative Decoding: The Idea": the small model guesses K
 * tokens one at a time; "CUDA Graphs: What They Are and Why They Helped":
 * the K steps replay as one graph): K greedy decode steps of the draft model. Writes the guesses
 * to the engine's device state and, when not NULL, to d_draft (device
 * [batch][K] int32) and their logits to d_logits (device [batch][K][vocab]
 * fp32). The first step runs two rows (the last two committed tokens) so the
 * draft cache always catches up with the committed sequence. With both
 * outputs NULL the K steps replay as one captured CUDA graph.
 */
SF_API sf_status sf_draft(sf_handle h, int32_t* d_draft, float* d_logits);

/*
 * Prompt-lookup draft ("Speculative decoding: correct, but slower (for
 * now)", Sangama page: guess what followed the last 2-4 tokens the last time
 * they appeared): for n = max_n down to min_n, the rightmost earlier
 * occurrence of the last n committed tokens; up to max_guess tokens that
 * followed it are proposed (cut at the end of the context). Optional device
 * outputs: d_prop [batch][max_guess] (unused slots 0), d_count [batch].
 * max_guess must be <= K.
 */
SF_API sf_status sf_ngram_draft(sf_handle h, int32_t max_guess, int32_t min_n, int32_t max_n,
                         int32_t* d_prop, int32_t* d_count);

/*
 * Several prompt-lookup guesses per round (the Sangama page, "Next": better
 * guesses for the look-back drafter; here several earlier occurrences are
 * checked by the target together instead of only the most recent one). The
 * earlier occurrences of the last n committed tokens are taken in
 * sf_ngram_draft's order (n from max_n down to min_n, rightmost first); each
 * gives up to g = K / n_cand tokens that followed it (cut at the end of the
 * context); a guess equal to one already taken is skipped; at most n_cand
 * guesses. Guess c fills verify rows 1 + c*g .. c*g + g. sf_verify then runs
 * the rows of each guess at the positions after the pending token, each
 * seeing the committed sequence and its own guess only, and
 * sf_accept_rollback takes the guess with the longest accepted prefix (the
 * lowest c on ties), commits as for one guess and moves that guess's
 * target-cache entries down to the committed slots. Optional device outputs:
 * d_prop [batch][n_cand][g] (unused 0), d_len [batch][n_cand] (0: no guess).
 * 1 <= n_cand <= K; 1 <= min_n <= max_n <= 64.
 */
SF_API sf_status sf_tree_draft(sf_handle h, int32_t n_cand, int32_t min_n, int32_t max_n, int32_t* d_prop,
                               int32_t* d_len);

/*
 * Target verify ("Speculative Decoding: The Idea": the target checks all
 * guesses in one forward pass; the Sangama page: the model's own choice at
 * every position): one causal pass over [pending, d_1..d_K] per sequence,
 * appending K+1 entries to the target cache. Optional device outputs: the
 * target's argmax at every row (d_tgt_argmax [batch][K+1] int32) and the
 * logits (d_logits [batch][K+1][vocab] fp32). Ties go to the lowest index.
 * With both outputs NULL the pass replays as one captured CUDA graph.
 */
SF_API sf_status sf_verify(sf_handle h, int32_t* d_tgt_argmax, float* d_logits);

/*
 * Accept and roll back ("Speculative Decoding: The Idea": keep the agreed
 * tokens; "Why It Kept Breaking (and How I Fixed It)", fix 4: in-place KV
 * rewind on rejection), per sequence: n = longest prefix of guesses equal to
 * the target's choices (capped at the number of real guesses); d_1..d_n and
 * the target's choice t_n are committed; both caches are cut back in place
 * to the committed length minus one. Host outputs (may be NULL):
 * h_n_accepted [batch], h_committed [batch][K+1], h_n_committed [batch].
 */
SF_API sf_status sf_accept_rollback(sf_handle h, int32_t* h_n_accepted, int32_t* h_committed,
                             int32_t* h_n_committed);

/* One whole round ("CUDA Graphs: What They Are and Why They Helped": one
 * driver call instead of a launch per kernel): draft (neural or n-gram, per
 * sf_set_drafter) + verify + accept/rollback as one CUDA graph replay. Host
 * outputs as in sf_accept_rollback (may be NULL). */
SF_API sf_status sf_step(sf_handle h, int32_t* h_n_committed, int32_t* h_committed);

/*
 * Run rounds until every sequence has at least n_new new tokens since its
 * prompt. The rounds run on the device as one graph launch: a WHILE
 * conditional node repeats the round graph, and a control kernel at the end
 * of each round decides on the device whether another round is needed and
 * fits in s_max (the pages' single driver call for the draft, "CUDA Graphs:
 * What They Are and Why They Helped", taken to the whole generation); the
 * host synchronises once. With SF_HOST_LOOP=1 in the environment at
 * sf_create the host replays the round graph instead, synchronising only to
 * count (same tokens). h_out: host [batch][n_new] (the first n_new generated
 * tokens). h_rounds: rounds run (may be NULL). SF_ERR_CAPACITY when s_max
 * runs out first.
 */
SF_API sf_status sf_generate(sf_handle h, int32_t n_new, int32_t* h_out, int32_t* h_rounds);

/* Rewind every sequence to its prompt (prefix already in the caches). */
SF_API sf_status sf_reset(sf_handle h);

/* Select the drafter used by sf_step / sf_generate (SF_DRAFT_*; min_n and
 * max_n apply to SF_DRAFT_NGRAM and SF_DRAFT_TREE only). */
SF_API sf_status sf_set_drafter(sf_handle h, int32_t mode, int32_t min_n, int32_t max_n);

/* Guesses per round of SF_DRAFT_TREE in sf_step / sf_generate (1..K; the
 * default is 2, or 1 when K = 1). */
SF_API sf_status sf_set_tree_candidates(sf_handle h, int32_t n_cand);

/* The guess each sequence's last multi-candidate round took (host [batch]). */
SF_API sf_status sf_tree_winner(sf_handle h, int32_t* h_c);

/* Current cache lengths per sequence (host [batch] each, may be NULL): the
 * positions the in-place rewind left ("Why It Kept Breaking", fixes 3-4:
 * explicit position updates, in-place rewind). */
SF_API sf_status sf_get_lengths(sf_handle h, int32_t* h_len_t, int32_t* h_len_d);

/* Accept-length histogram since prefill: host [batch][K+1]. */
SF_API sf_status sf_get_accept_hist(sf_handle h, int32_t* h_hist);

/*
 * Launch timeline, for profiling. Only when the environment variable
 * SF_TRACE=1 was set at sf_create: every kernel of the forward passes
 * stamps the GPU global timer (ns) when it starts and when its wait on the
 * preceding kernel returns. sf_trace copies up to max_launches pairs
 * {start, wait_done} into h_out (host, 2 x uint64 each) for launch slots
 * 0.. (launch n uses slot n mod 8192; graph replays rewrite their slots) and
 * returns the count; with h_out NULL it returns the number of launches
 * enqueued so far; 0 when tracing is off. sf_trace_label(i) names slot i ("qkv",
 * "attention", "merge", "o_proj", "gate_up", "down", "lm_head", "embed").
 */
SF_API int32_t sf_trace(sf_handle h, uint64_t* h_out, int32_t max_launches);
SF_API const char* sf_trace_label(sf_handle h, int32_t i);

/* Kernel launches in one round of the current drafter (the node count of
 * its round graph; every node is a kernel; sf_generate's device loop adds one
 * control kernel per round), or 0 before a round graph has been built by
 * sf_step / sf_generate. */
SF_API int64_t sf_round_launches(sf_handle h);

/* Name of a status code; message of the calling thread's last failure. */
SF_API const char* sf_status_str(sf_status s);
SF_API const char* sf_last_error(void);
/* Release the engine's graphs, stream and pinned host memory (the caller's
 * device buffers stay the caller's). NULL is ignored. */
SF_API void sf_destroy(sf_handle h);

/*
 * One skinny linear map on its own: y[m][n] = sum_k x[m][k] * W[n][k] for
 * m < M (1..SF_MAX_ROWS), the weight-streaming GEMM every projection of the
 * forward pass uses. W: device bf16 [N, ld] row-major (ld >= K, K and ld
 * multiples of 8, 16-byte aligned rows); x: device fp32 [M, K]; y: device
 * fp32 [M, N]. d_workspace: device scratch of
 * sf_linear_workspace_bytes(N, K) bytes, 256-byte aligned, for split-K
 * partial tiles, arrival counters (zeroed by the call) and a bf16 hi/lo copy
 * of x in the GEMM's operand order. Enqueued on cuda_stream; returns without
 * synchronising. There is no device status word here: should a weight-tile
 * wait ever expire, the kernel returns normally and y is unspecified.
 */
SF_API size_t sf_linear_workspace_bytes(int32_t N, int32_t K);
SF_API sf_status sf_linear(const void* d_w, int32_t N, int32_t K, int32_t ld, const float* d_x, int32_t M,
                           float* d_y, void* d_workspace, void* cuda_stream);

/*
 * The two halves of sf_linear. Every projection reads its token rows in the
 * order its GEMM kernel consumes them.
 * Up to 16 rows ("fragment order", the mma.sync kernel): bf16 pairs (hi =
 * bf16(v), lo = bf16(v - hi), about 16 mantissa bits of the fp32 value) in
 * the order the MMA lanes read their B operand: with T = ceil(M / 4) token
 * tiles, the 16-byte unit ((j * T + t) * 2 + h) * 32 + l holds, for 64-feature
 * chunk j, tile t, half h and lane l = 4 * col + c, the 8 features
 * 64j + 16c + 8h + 0..7 of token 4t + col / 2, hi parts for even col and lo
 * parts for odd col.
 * More than 16 rows (the tcgen05 kernel; the threshold is 17 unless
 * SF_UMMA_MIN_ROWS says otherwise): bf16(v) in the tensor-core B tile with
 * 128-byte swizzle: with T8 = ceil(M / 8), the 1024-byte block at byte
 * (j * T8 + t) * 1024 holds tokens 8t .. 8t+7 of chunk j, one 128-byte row
 * per token (row m % 8), its 16-byte piece q (features 64j + 8q .. +7) at
 * position q ^ (m % 8) of the row.
 * Features past K and tokens past M are zero.
 *   sf_frag_bytes(K, M): size of the copy to allocate (0 if invalid).
 *   sf_to_frag: x (device fp32 [M, ld], features 0..K-1) -> d_frag (device,
 *     16-byte aligned, sf_frag_bytes(K, M) bytes), enqueued on cuda_stream.
 *   sf_linear_frag: sf_linear reading the copy instead of x (same W, y and
 *     workspace rules); reuse one copy for several matrices that share x.
 */
SF_API size_t sf_frag_bytes(int32_t K, int32_t M);
SF_API sf_status sf_to_frag(const float* d_x, int32_t M, int32_t K, int32_t ld, void* d_frag, void* cuda_stream);
SF_API sf_status sf_linear_frag(const void* d_w, int32_t N, int32_t K, int32_t ld, const void* d_frag, int32_t M,
                                float* d_y, void* d_workspace, void* cuda_stream);

/*
 * sf_linear without any caller-provided scratch, for callers that cannot
 * allocate device memory where they need the projection: plug-ins whose
 * host framework owns every device allocation through its own pool, and
 * latency-critical loops that cannot afford cudaMalloc's implicit device
 * synchronisation. Same arguments and result as sf_linear minus d_workspace.
 * (The pages have no counterpart of this call.)
 *
 * The scratch is a file-scope device array of about 38 MB inside the
 * library, enough for N up to 1,048,576 output rows, K up to 65,536 inputs
 * and M up to SF_MAX_ROWS token rows; every GPU that loads the library keeps
 * it until the process exits. The call allocates nothing: the first call on
 * each device looks up the array's device address (cudaGetSymbolAddress)
 * with that device current and keeps it for the life of the process, so a
 * context reset (cudaDeviceReset) after that first call is not supported.
 * All calls share the array: it keeps the last call's contents, the counters
 * that must start at zero are cleared by each call, and calls that overlap
 * on the GPU race with each other. N, K or M beyond the limits returns
 * SF_ERR_ARG with a message in sf_last_error().
 */
SF_API sf_status sf_linear_noalloc(const void* d_w, int32_t N, int32_t K, int32_t ld, const float* d_x,
                                   int32_t M, float* d_y, void* cuda_stream);

/*
 * Blockwise NF4 quantisation of a bf16 matrix on the device (a preparation
 * step for SF_WDTYPE_NF4 weights): w [rows, cols] with row stride ld
 * elements, cols a multiple of 64; writes packed codes [rows, cols/2] and fp16
 * block scales [rows, 8 * ceil(cols / 512)] (padding entries untouched).
 * Codebook: the NormalFloat construction of
 * Dettmers et al., "QLoRA" (2023), section 3 (format named in "The Numbers").
 */
SF_API sf_status sf_nf4_quantize(const void* d_w, int32_t rows, int32_t cols, int32_t ld,
                          void* d_packed, void* d_scales, void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* SF_H_ */
