// Host side of the engine: the C ABI declared in include/sf.h.
//
// The engine binds caller-owned device buffers, plans every GEMM once (row
// blocks, K split) from the matrix shape and the SM count, and enqueues the
// forward passes of the draft and target models. All lengths, positions and
// tokens of the speculative round live on the device, so one round is a
// fixed sequence of launches: it is captured once into a CUDA graph per
// drafter and replayed with no host writes in between ("CUDA Graphs: What
// They Are and Why They Helped" and "Why It Kept Breaking (and How I Fixed
// It)", I Got 28 TPS Out of Free Kaggle GPUs: static cache, in-place
// buffers, positions updated on the device, in-place rewind).
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "sf_kernels.h"

using namespace sf;

namespace {

thread_local std::string g_err;

sf_status fail(sf_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

#define CK(x)                                                                                   \
  do {                                                                                          \
    cudaError_t e_ = (x);                                                                       \
    if (e_ != cudaSuccess)                                                                      \
      return fail(SF_ERR_CUDA, "%s failed: %s (%s:%d)", #x, cudaGetErrorString(e_), __FILE__, \
                  __LINE__);                                                                    \
  } while (0)

struct Plan {
  int nblocks = 0, nsplit = 1, cps = 1;
  int cluster = 1;   // the K slices of a row block form one cluster (else: global partial tiles)
};

// Split K only when the row blocks alone cannot fill the GPU; the split
// depends on the matrix shape and the SM count, never on the number of
// token rows, so every row is computed the same way in every launch.
Plan make_plan(int nblocks, int K, int slots, int max_split, int cps_align = 1) {
  Plan p;
  p.nblocks = nblocks;
  const int nch = (K + kChunk - 1) / kChunk;
  int ns = 1;
  if (nblocks * 10 < slots * 9) ns = std::max(1, slots / nblocks);
  ns = std::min(std::min(ns, nch), max_split);
  p.cps = (nch + ns - 1) / ns;
  p.cps = (p.cps + cps_align - 1) / cps_align * cps_align;   // NF4 slices start on 4-chunk groups
  p.nsplit = (nch + p.cps - 1) / p.cps;
  return p;
}

enum { W_Q = 0, W_K, W_V, W_O, W_G, W_U, W_D };

struct LayerW {
  CUtensorMap tm[7];
  CUtensorMap tms[7];      // NF4 block scales
  CUtensorMap tmu[7];      // the same with 64-row boxes, for the tcgen05 GEMM (forwards of > 16 rows)
  CUtensorMap tmsu[7];
  const void* w[7] = {};
  const void* sc[7] = {};  // NF4 block scales
  const void *ln1 = nullptr, *ln2 = nullptr, *bq = nullptr, *bk = nullptr, *bv = nullptr;   // bf16 or fp32
};

struct Model {
  sf_model_cfg c{};
  const void* embed = nullptr;   // bf16, or fp32 (SF_WDTYPE_F32)
  int embed_ld = 0;
  std::vector<LayerW> L;
  const void* norm = nullptr;
  const void* lm = nullptr;
  int lm_ld = 0;
  CUtensorMap lm_tm;
  CUtensorMap lm_tmu;      // 64-row boxes: the LM head of forwards of more than 16 rows (tcgen05)
  bf16* kv = nullptr;
  CUtensorMap kvmap;       // the whole cache as [rows][head_dim] for the attention kernel's TMA
  CUtensorMap kvmap8;      // the same with 8-slot boxes
  int attn_R = 1;          // cache chunks per attention work item
  int attn_stages = 1;     // key/value chunks in flight per attention CTA
  bool attn_group = false; // attention items carry up to four query tiles (else one)
  int dec_rows = 0;        // forwards of at most this many rows (<= 4) run as one persistent kernel (k_decode)
  DecLayer* dlay = nullptr;   // its device table of layer pointers
  float2* rope = nullptr;
  Plan p_qkv, p_o, p_gu, p_d, p_lm;
  Plan u_qkv, u_o, u_gu, u_d, u_lm;   // tcgen05 GEMM plans (forwards of more than 16 rows)
  int q_dim() const { return c.n_heads * c.head_dim; }
  int kv_dim() const { return c.n_kv_heads * c.head_dim; }
};

// sf_linear's split-K scratch: partial tiles of 16 token rows x 128 outputs
// (row blocks x K slices x row groups).
constexpr int kLinearTiles = 2048;
constexpr size_t kLinearPartBytes = (size_t)kLinearTiles * kGroupRows * kBlockRows * 4;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

constexpr int kMaxSms = 256;   // bound on the SM count for workspace sizing

bool cfg_ok(const sf_model_cfg* c, std::string* why) {
  auto bad = [&](const char* m) {
    *why = m;
    return false;
  };
  if (!c) return bad("null model config");
  if (c->layers < 1 || c->hidden < 128 || c->n_heads < 1 || c->n_kv_heads < 1 || c->ffn < 8 ||
      c->vocab < 1)
    return bad("non-positive dimension");
  if (c->hidden % 128) return bad("hidden must be a multiple of 128");
  if (c->head_dim != 64 && c->head_dim != 128) return bad("head_dim must be 64 or 128");
  if (c->n_heads % c->n_kv_heads) return bad("n_heads must be a multiple of n_kv_heads");
  if ((c->n_heads * c->head_dim) % 128 || (c->n_kv_heads * c->head_dim) % 128)
    return bad("n_heads*head_dim and n_kv_heads*head_dim must be multiples of 128");
  if (c->ffn % 8) return bad("ffn must be a multiple of 8");
  if (c->wdtype != SF_WDTYPE_BF16 && c->wdtype != SF_WDTYPE_NF4 && c->wdtype != SF_WDTYPE_F32)
    return bad("unknown wdtype");
  if (c->wdtype == SF_WDTYPE_NF4 && c->ffn % 64) return bad("NF4 weights need ffn to be a multiple of 64");
  const int eld = c->embed_ld ? c->embed_ld : c->hidden;
  if (eld < c->hidden || eld % 8) return bad("embed_ld must be >= hidden and a multiple of 8");
  if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f)) return bad("bad rms_eps or rope_theta");
  return true;
}

struct Layout {
  size_t x, ssq, q, apart, upart, counters, keys, done, zeros, fx, fh, fo, fa, rope_t, rope_d, state, trace, dh, dbar,
      dlay_t, dlay_d, total;
  int n_kv_chunks, max_blocks;
};

int nblocks_of(const sf_model_cfg* c, int which) {
  switch (which) {
    case 0: return (c->n_heads * c->head_dim + 2 * c->n_kv_heads * c->head_dim + 127) / 128;
    case 1: return (c->hidden + 127) / 128;
    case 2: return (c->ffn + 63) / 64;
    default: return (c->vocab + 127) / 128;
  }
}

// State ints: len_t, len_d, vtok, ttok, dtok0, nprop, hist, prompt_len,
// acc_hist, then the report block (ncommit, nacc, commit, total, err) that
// one copy brings back to the host.
struct StateOff {
  size_t len_t, len_d, vtok, ttok, dtok0, nprop, hist, prompt_len, acc_hist, loop_target, clen, report, ncommit,
      nacc, commit, total, err, rounds, tree_c, n_ints, report_ints;
};

StateOff state_offsets(int B, int K, int s_max) {
  StateOff o{};
  size_t p = 0;
  auto take = [&](size_t n) {
    size_t r = p;
    p += (n + 63) & ~size_t(63);
    return r;
  };
  const int K1 = K + 1;
  o.len_t = take(B);
  o.len_d = take(B);
  o.vtok = take(B * K1);
  o.ttok = take(B * K1);
  o.dtok0 = take(2 * B);
  o.nprop = take(B);
  o.hist = take((size_t)B * s_max);
  o.prompt_len = take(B);
  o.acc_hist = take(B * K1);
  o.loop_target = take(1);
  o.clen = take(B * K);
  o.report = p;
  o.ncommit = p;
  p += B;
  o.nacc = p;
  p += B;
  o.commit = p;
  p += B * K1;
  o.total = p;
  p += B;
  o.err = p;
  p += 1;
  o.rounds = p;
  p += 1;
  o.tree_c = p;
  p += B;
  o.report_ints = p - o.report;
  o.n_ints = p;
  return o;
}

Layout make_layout(const sf_model_cfg* t, const sf_model_cfg* d, int B, int K, int s_max) {
  Layout L{};
  auto mx = [&](auto f) { return d ? std::max(f(t), f(d)) : f(t); };
  const int H = mx([](const sf_model_cfg* c) { return c->hidden; });
  const int QD = mx([](const sf_model_cfg* c) { return c->n_heads * c->head_dim; });
  const int NQ = mx([](const sf_model_cfg* c) { return c->n_heads; });
  const int HD = mx([](const sf_model_cfg* c) { return c->head_dim; });
  const int F = mx([](const sf_model_cfg* c) { return c->ffn; });
  L.n_kv_chunks = s_max / kKvChunk;
  L.max_blocks = 0;
  for (int w = 0; w < 4; ++w) L.max_blocks = std::max(L.max_blocks, mx([w](const sf_model_cfg* c) { return nblocks_of(c, w); }));
  size_t p = 0;
  auto take = [&](size_t bytes) {
    size_t r = p;
    p = align256(p + bytes);
    return r;
  };
  L.x = take((size_t)kRows * H * 4);
  L.ssq = take((size_t)(H / 128) * kRows * 4);
  L.q = take((size_t)kRows * QD * 4);
  L.apart = take((size_t)kRows * NQ * L.n_kv_chunks * (HD + 2) * 4);
  // tcgen05 GEMM partial tiles when its K slices cannot all be clusters: at
  // most two CTAs per SM, each with up to SF_MAX_ROWS x 128 floats.
  L.upart = take((size_t)2 * kMaxSms * kRows * kBlockRows * 4);
  L.counters = take((size_t)L.max_blocks * kMaxGroups * 4);
  L.keys = take((size_t)kRows * 8);
  L.done = take(4);
  L.zeros = take((size_t)B * 4);
  // Fragment-ordered GEMM inputs (zeroed at creation: features past K stay 0):
  // normed residual for QKV / LM head, normed residual for gate/up,
  // attention output, SwiGLU activation.
  const int kTiles = (kRows + 3) / 4;
  L.fx = take(frag_bytes(H, kTiles));
  L.fh = take(frag_bytes(H, kTiles));
  L.fo = take(frag_bytes(QD, kTiles));
  L.fa = take(frag_bytes(F, kTiles));
  L.rope_t = take((size_t)s_max * (t->head_dim / 2) * 8);
  L.rope_d = d ? take((size_t)s_max * (d->head_dim / 2) * 8) : p;
  L.state = take(state_offsets(B, K, s_max).n_ints * 4);
  L.trace = take((size_t)2 * 8192 * 8);
  // The persistent decode forward: SwiGLU output of up to 4 rows, its grid
  // barrier words, and each model's table of layer pointers.
  L.dh = take((size_t)4 * F * 4);
  L.dbar = take(16 + (size_t)4 * 64 * 4);   // barrier words + per-(sequence, KV head) counters
  L.dlay_t = take((size_t)t->layers * sizeof(DecLayer));
  L.dlay_d = d ? take((size_t)d->layers * sizeof(DecLayer)) : p;
  L.total = p;
  return L;
}

}  // namespace

sf_status sf::set_error(sf_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

struct sf_engine {
  Model tgt, dft;
  bool has_dft = false;
  bool pdl = true;      // programmatic dependent launch between the round's kernels
  bool dec_on = false;  // SF_PERSISTENT=1: forwards of at most 4 rows run as one persistent kernel
  bool box8 = false;    // SF_KV_BOX8=1: attention loads a partly filled chunk in 8-slot boxes
  float* dh = nullptr;       // persistent decode: SwiGLU output
  unsigned* dbar = nullptr;  // persistent decode: grid barrier words
  bool expire_waits = false;   // SF_TEST_WAIT_EXPIRE=1: every GEMM reports an expired wait (error-path test)
  unsigned long long* trace = nullptr;     // launch timeline (SF_TRACE=1), kTraceSlots entries
  int trace_next = 0;
  std::vector<std::string> trace_labels;
  int B = 0, K = 0, s_max = 0, num_sms = 0, slots = 0;
  cudaStream_t user = nullptr, cap = nullptr;
  unsigned char* ws = nullptr;
  float* upart = nullptr;   // tcgen05 GEMM partial tiles (non-cluster K split)
  Layout lay{};
  StateOff so{};
  bf16 *fx = nullptr, *fh = nullptr, *fo = nullptr, *fa = nullptr;
  float *x = nullptr, *ssq = nullptr, *q = nullptr, *apart = nullptr;
  int *counters = nullptr, *done = nullptr, *zeros = nullptr;
  unsigned long long* keys = nullptr;
  SpecState st{};
  int* pin = nullptr;   // pinned host copy of the report block
  cudaGraphExec_t graph[4] = {};   // whole round, per drafter (SF_DRAFT_*)
  size_t graph_kernels[4] = {};    // kernel launches in each round graph
  cudaGraphExec_t loop[4] = {};    // sf_generate: rounds in a device-side WHILE loop
  bool host_loop = false;   // SF_HOST_LOOP=1: sf_generate replays the round graph from the host instead
  cudaGraphExec_t g_draft = nullptr, g_verify = nullptr, g_verify_tree = nullptr;
  int g_verify_tree_g = 0;   // guesses per candidate g_verify_tree was captured with
  int drafter = SF_DRAFT_NEURAL, ng_min = 2, ng_max = 4;
  int tree_n = 1;            // SF_DRAFT_TREE: candidates per round (g = K / tree_n guesses each)
  int drafted_tree_n = 1;    // candidates of the last sf_tree_draft
  std::vector<int> C;   // committed tokens per sequence (host mirror)
  std::vector<int> P;   // prompt length per sequence
  int phase = 0;        // 0: no prompt, 1: ready, 2: drafted, 3: verified
  int drafted_mode = SF_DRAFT_NEURAL;
  bool draft_stale = false;
};

namespace {

sf_status bind_model(sf_engine* e, Model& md, const sf_model_cfg* c, const void* const* w, bf16* kv) {
  md.c = *c;
  // Null is allowed only for biases of a bias-free config; every pointer must
  // be 16-byte aligned (the kernels read rows with 128-bit loads).
  auto check = [](const void* p, const char*, bool allow_null) -> bool {
    if (!p) return allow_null;
    return (reinterpret_cast<uintptr_t>(p) & 15) == 0;
  };
  int i = 0;
  md.embed = w[i++];
  if (!check(md.embed, "embed", false)) return fail(SF_ERR_ARG, "embed pointer null or not 16-byte aligned");
  md.embed_ld = c->embed_ld ? c->embed_ld : c->hidden;
  md.L.resize(c->layers);
  const bool nf4 = c->wdtype == SF_WDTYPE_NF4;
  for (int l = 0; l < c->layers; ++l) {
    LayerW& lw = md.L[l];
    // NF4: every linear map is two slots, packed codes then block scales.
    auto lin = [&](int k) {
      lw.w[k] = w[i++];
      if (nf4) lw.sc[k] = w[i++];
    };
    lw.ln1 = w[i++];
    lin(W_Q);
    lin(W_K);
    lin(W_V);
    lw.bq = w[i++];
    lw.bk = w[i++];
    lw.bv = w[i++];
    lin(W_O);
    lw.ln2 = w[i++];
    lin(W_G);
    lin(W_U);
    lin(W_D);
    if (!c->qkv_bias) lw.bq = lw.bk = lw.bv = nullptr;
    bool ok = check(lw.ln1, "ln1", false) && check(lw.ln2, "ln2", false);
    for (int k = 0; k < 7; ++k) ok = ok && check(lw.w[k], "w", false) && (!nf4 || check(lw.sc[k], "scales", false));
    if (c->qkv_bias) ok = ok && check(lw.bq, "bq", false) && check(lw.bk, "bk", false) && check(lw.bv, "bv", false);
    if (!ok) return fail(SF_ERR_ARG, "layer %d: a weight pointer is null or not 16-byte aligned", l);
  }
  md.norm = w[i++];
  if (!check(md.norm, "norm", false)) return fail(SF_ERR_ARG, "final norm pointer null or misaligned");
  if (c->tied) {
    md.lm = md.embed;
    md.lm_ld = md.embed_ld;
  } else {
    md.lm = w[i++];
    md.lm_ld = c->hidden;
    if (!check(md.lm, "lm_head", false)) return fail(SF_ERR_ARG, "lm_head pointer null or misaligned");
  }
  md.kv = kv;
  {
    const long rows = (long)c->layers * 2 * e->B * c->n_kv_heads * e->s_max;
    cudaError_t ce = make_kv_map(&md.kvmap, kv, rows, c->head_dim);
    if (ce == cudaSuccess) ce = make_kv_map(&md.kvmap8, kv, rows, c->head_dim, 8);
    if (ce != cudaSuccess) return fail(SF_ERR_CUDA, "KV cache tensor map: %s", cudaGetErrorString(ce));
    // Attention work items of R chunks: one chunk each while the cache is
    // small; up to 8 for a large batch of long caches, so the items fill the
    // GPU a few times over and the merge reads a few partials per row. Fixed
    // per model and engine: a row's arithmetic never depends on other rows.
    // The same load decides how many chunks a CTA keeps in flight, and
    // whether an item carries every query tile of its KV head (each chunk
    // read once) or one tile (more items for a small batch: the same work
    // spread over more CTAs; measured faster for the batch-1 verify).
    const long load = (long)e->B * c->n_kv_heads * (e->s_max / kKvChunk) / 2048;
    md.attn_R = load >= 8 ? 8 : (load >= 4 ? 4 : (load >= 2 ? 2 : 1));
    md.attn_stages = load >= 2 ? 2 : 1;
    md.attn_group = load >= 2;
    // SF_ATTN_R (chunks per range, 1..16) and SF_ATTN_STAGES (1 or 2)
    // override the choice, for tuning; results depend on R only.
    if (const char* v = getenv("SF_ATTN_R")) md.attn_R = std::min(16, std::max(1, atoi(v)));
    if (const char* v = getenv("SF_ATTN_STAGES")) md.attn_stages = atoi(v) == 2 ? 2 : 1;
  }
  const int H = c->hidden;
  const int QD = c->n_heads * c->head_dim, KVD = c->n_kv_heads * c->head_dim, F = c->ffn;
  const bool f32 = c->wdtype == SF_WDTYPE_F32;   // plain pointers, no tensor maps
  for (int l = 0; l < c->layers && !f32; ++l) {
    LayerW& lw = md.L[l];
    const int rows[7] = {QD, KVD, KVD, H, F, F, H};
    const int ks[7] = {H, H, H, QD, H, H, F};
    for (int k = 0; k < 7; ++k) {
      cudaError_t ce = nf4 ? make_nf4_maps(&lw.tm[k], &lw.tms[k], lw.w[k], lw.sc[k], rows[k], ks[k])
                           : make_weight_map(&lw.tm[k], lw.w[k], rows[k], ks[k], ks[k]);
      if (ce == cudaSuccess)
        ce = nf4 ? make_nf4_maps(&lw.tmu[k], &lw.tmsu[k], lw.w[k], lw.sc[k], rows[k], ks[k], 64)
                 : make_weight_map(&lw.tmu[k], lw.w[k], rows[k], ks[k], ks[k], 64);
      if (ce != cudaSuccess)
        return fail(SF_ERR_CUDA, "layer %d weight %d: tensor map: %s", l, k, cudaGetErrorString(ce));
    }
  }
  if (!f32) {
    cudaError_t ce = make_weight_map(&md.lm_tm, md.lm, c->vocab, H, md.lm_ld);
    if (ce == cudaSuccess) ce = make_weight_map(&md.lm_tmu, md.lm, c->vocab, H, md.lm_ld, 64);
    if (ce != cudaSuccess) return fail(SF_ERR_CUDA, "LM head tensor map: %s", cudaGetErrorString(ce));
  }
  // The K splits of a row block form one thread-block cluster. Matrices of
  // 24 MB and more are split for two CTAs per SM (bandwidth) in clusters of
  // at most 8 (the portable size, which packs well into GPCs); smaller ones
  // for one CTA per SM in clusters of up to 16, so that the next kernel's
  // CTAs fit beside them and start streaming early. Clusters are placed
  // within GPCs, and a kernel's CTAs start while the preceding kernel still
  // holds part of the GPU: the split is lowered until the clusters fit with a
  // fifth of the cluster slots to spare (checked for the 9..12-row
  // footprint), so that fragmented free space still takes them all.
  const int al = nf4 ? 4 : 1;
  auto plan = [&](int nblocks, long rows, long k) {
    const bool big = rows * k * (nf4 ? 1 : 2) >= (24l << 20);
    const int slots = big ? 2 * e->num_sms : e->num_sms;
    // Matrices of 64 MB and more whose row blocks fill less than a third of
    // the CTA slots take more than 8 K slices, summed through global partial
    // tiles (the last CTA of a row block adds them in order): bandwidth over
    // the cluster reduction's lower latency.
    if (rows * k * (nf4 ? 1 : 2) >= (64l << 20) && slots / nblocks > 8) {
      Plan p = make_plan(nblocks, (int)k, slots, 16, al);
      if (p.nsplit > 8) {
        p.cluster = 0;
        return p;
      }
    }
    Plan p = make_plan(nblocks, (int)k, slots, big ? 8 : kMaxClusterSplit, al);
    while (p.nsplit > 1) {
      const int stages = pick_stages(p.nblocks * p.nsplit, p.cps, e->num_sms, nf4);
      if (5 * p.nblocks <= 4 * gemm_max_clusters(p.nsplit, 12, stages, p.cps)) break;
      p = make_plan(nblocks, (int)k, slots, p.nsplit - 1, al);
    }
    return p;
  };
  const long QKV = (long)c->n_heads * c->head_dim + 2l * c->n_kv_heads * c->head_dim;
  md.p_qkv = plan(nblocks_of(c, 0), QKV, H);
  md.p_o = plan(nblocks_of(c, 1), H, (long)c->n_heads * c->head_dim);
  md.p_gu = plan(nblocks_of(c, 2), 2l * c->ffn, H);
  md.p_d = plan(nblocks_of(c, 1), H, c->ffn);
  // tcgen05 GEMM: two CTAs per SM whatever the row count, up to 8 K slices;
  // the slices of a row block form a cluster when all clusters fit on the GPU
  // at once, else they add their tiles through global memory (the cluster
  // placement of this footprint allows far fewer than two CTAs per SM).
  auto uplan = [&](int nblocks, long k) {
    const int stages = umma_stages(kRows, nf4);
    Plan p = make_plan(nblocks, (int)k, 2 * e->num_sms, 8, al);
    if (p.nsplit > 1 && p.nblocks > umma_max_clusters(p.nsplit, kRows, stages, nf4)) p.cluster = 0;
    return p;
  };
  md.u_qkv = uplan(nblocks_of(c, 0), H);
  md.u_o = uplan(nblocks_of(c, 1), (long)c->n_heads * c->head_dim);
  md.u_gu = uplan(nblocks_of(c, 2), H);
  md.u_d = uplan(nblocks_of(c, 1), c->ffn);
  md.u_lm.nblocks = nblocks_of(c, 3);   // LM heads: no K split
  md.u_lm.nsplit = 1;
  md.u_lm.cps = (H + kChunk - 1) / kChunk;
  md.p_lm.nblocks = nblocks_of(c, 3);   // the persistent LM head: no K split
  md.p_lm.nsplit = 1;
  md.p_lm.cps = (H + kChunk - 1) / kChunk;
  return SF_OK;
}

GemmArgs base_args(sf_engine* e, const Model& md, const Plan& p, const RowSet& rs) {
  GemmArgs a{};
  a.nblocks = p.nblocks;
  a.nsplit = p.nsplit;
  a.cps = p.cps;
  a.stages = pick_stages(p.nblocks * p.nsplit, p.cps, e->num_sms);
  a.counter = e->counters;
  a.cluster = 1;   // the K slices of a row block are one cluster
  a.err = e->st.err;
  a.wf32 = md.c.wdtype == SF_WDTYPE_F32 ? 1 : 0;
  a.expire_first_wait = e->expire_waits ? 1 : 0;
  a.rs = rs;
  a.eps = md.c.rms_eps;
  return a;
}


// Give the next launch a timeline slot (when tracing) and remember its name.
RowSet traced(sf_engine* e, RowSet rs, const char* what) {
  rs.trace = e->trace;
  if (e->trace) {
    rs.trace_id = e->trace_next % kTraceSlots;
    if ((int)e->trace_labels.size() <= rs.trace_id) e->trace_labels.resize(rs.trace_id + 1);
    e->trace_labels[rs.trace_id] = what;
    ++e->trace_next;
  }
  return rs;
}

struct TokOut {
  int* tok = nullptr;
  int stride = 0, skip = 0, off = 0;
  float* logits = nullptr;
  int lg_stride = 0, lg_off = 0;
};

// Enqueue one forward pass of `md` over the rows `rs`. With `lm` the final
// norm + LM head + argmax run too and write tokens (and optional logits).
// seq >= 0: every row belongs to sequence `seq` alone (its cache is addressed
// as a batch of one; rs.pos_base then has one entry).
sf_status forward(sf_engine* e, Model& md, const RowSet& rs, bool lm, const TokOut& to, cudaStream_t s,
                  int seq = -1) {
  const sf_model_cfg& c = md.c;
  const int nf4 = c.wdtype == SF_WDTYPE_NF4 ? 1 : 0;
  const int H = c.hidden, QD = md.q_dim(), KVD = md.kv_dim();
  // More than 16 token rows: the projections run on the tcgen05 GEMM, whose
  // inputs the producers write in the tensor-core operand order (the LM head
  // keeps reading fragment order).
  const bool f32 = c.wdtype == SF_WDTYPE_F32;   // fp32 weights: the plain fp32 kernel, fragment order
  const bool tc = !f32 && rs.M >= (nf4 ? umma_min_rows_nf4() : umma_min_rows());
  auto gemm = [&](const GemmArgs& a, int epi) {
    if (f32) return launch_gemm_f32(a, epi, s, e->pdl);
    return tc ? launch_umma(a, epi, s, e->pdl) : launch_gemm(a, epi, s, e->pdl);
  };
  auto maps = [&](GemmArgs& a, const LayerW& lw, int slot, int w) {
    a.tm[slot] = tc ? lw.tmu[w] : lw.tm[w];
    a.tms[slot] = tc ? lw.tmsu[w] : lw.tms[w];
  };
  auto stages = [&](const GemmArgs& a) {
    return tc ? umma_stages(rs.M, nf4) : pick_stages(a.nblocks * a.nsplit, a.cps, e->num_sms, nf4);
  };
  auto uplan_args = [&](GemmArgs& a, const Plan& p) {   // cluster or global K-slice sums
    a.cluster = p.cluster;
    a.part = e->upart;
  };
  // At most four rows (a decode step): one persistent kernel for the whole
  // forward up to the LM head's input.
  const bool use_dec = e->dec_on && rs.M <= md.dec_rows && rs.rps <= 2 && rs.tree_g == 0 && seq < 0;
  if (use_dec) {
    DecArgs d{};
    d.layers = md.dlay;
    d.L = c.layers;
    d.H = H;
    d.nq = c.n_heads;
    d.nkv = c.n_kv_heads;
    d.hd = c.head_dim;
    d.F = c.ffn;
    d.vocab = c.vocab;
    d.embed = static_cast<const bf16*>(md.embed);
    d.embed_ld = md.embed_ld;
    d.norm = static_cast<const bf16*>(md.norm);
    d.eps = c.rms_eps;
    d.scale = 1.0f / sqrtf((float)c.head_dim);
    d.rope = md.rope;
    d.kv = md.kv;
    d.B = e->B;
    d.s_max = e->s_max;
    d.R = 1;
    d.n_ranges = e->lay.n_kv_chunks;
    d.x = e->x;
    d.q = e->q;
    d.part = e->apart;
    d.h = e->dh;
    d.frag = e->fx;
    d.ssq = e->ssq;
    d.bar = e->dbar;
    d.cnt = e->dbar + 4;
    d.err = e->st.err;
    d.expire_first_wait = e->expire_waits ? 1 : 0;
    d.rs = traced(e, rs, "decode");
    // Timeline slots of the kernel's phases, right after its own (which the
    // embedding phase stamps).
    if (e->trace)
      for (int l = 0; l < c.layers; ++l)
        for (const char* ph : {"d_qkv", "d_attention", "d_o_proj", "d_gate_up", "d_down"}) traced(e, rs, ph);
    CK(launch_decode(d, e->num_sms, s));
  }
  EmbedArgs ea{};
  ea.E = md.embed;
  ea.ld = md.embed_ld;
  ea.H = H;
  ea.vocab = c.vocab;
  ea.err = e->st.err;
  ea.x = e->x;
  ea.ssq = e->ssq;
  ea.frag = e->fx;
  ea.gain = md.L[0].ln1;
  ea.f32 = f32;
  ea.umma = tc;
  if (!use_dec) {
    ea.rs = traced(e, rs, "embed");
    CK(launch_embed(ea, s, e->pdl));
    const size_t seq_elems = (size_t)c.n_kv_heads * e->s_max * c.head_dim;   // one sequence's keys of a layer
    const size_t layer_elems = 2 * e->B * seq_elems;
    for (int l = 0; l < c.layers; ++l) {
      const LayerW& lw = md.L[l];
      bf16* kc = md.kv + (size_t)l * layer_elems;
      bf16* vc = kc + layer_elems / 2;
      if (seq >= 0) {
        kc += seq * seq_elems;
        vc += seq * seq_elems;
      }
      // q, k, v (+ bias, RoPE, cache append)
      GemmArgs a = base_args(e, md, tc ? md.u_qkv : md.p_qkv, rs);
      a.w[0] = lw.w[W_Q];
      a.w[1] = lw.w[W_K];
      a.w[2] = lw.w[W_V];
      maps(a, lw, 0, W_Q);
      maps(a, lw, 1, W_K);
      maps(a, lw, 2, W_V);
      a.nf4 = nf4;
      a.stages = stages(a);
      uplan_args(a, tc ? md.u_qkv : md.p_qkv);
      a.bias[0] = lw.bq;
      a.bias[1] = lw.bk;
      a.bias[2] = lw.bv;
      a.seg_end[0] = QD;
      a.seg_end[1] = QD + KVD;
      a.seg_end[2] = QD + 2 * KVD;
      a.ld[0] = a.ld[1] = a.ld[2] = H;
      a.nseg = 3;
      a.N = QD + 2 * KVD;
      a.K = H;
      a.in = reinterpret_cast<const uint4*>(e->fx);
      a.ssq = e->ssq;
      a.nssq = H / 128;
      a.inv_k = 1.0f / H;
      a.out = e->q;
      a.out_ld = QD;
      a.q_dim = QD;
      a.kv_dim = KVD;
      a.hd = c.head_dim;
      a.nkv = c.n_kv_heads;
      a.s_max = e->s_max;
      a.kc = kc;
      a.vc = vc;
      a.rope = md.rope;
      a.rs = traced(e, rs, "qkv");
      CK(gemm(a, EPI_QKV));
      // attention
      AttnArgs t{};
      t.kvmap = md.kvmap;
      t.kvmap8 = md.kvmap8;
      t.kc = kc;
      t.vc = vc;
      t.box8 = e->box8 ? 1 : 0;
      t.kv_brows = c.n_kv_heads * e->s_max;
      t.kv_vrows = e->B * t.kv_brows;
      t.kv_row0 = (2 * l * e->B + (seq >= 0 ? seq : 0)) * t.kv_brows;
      t.R = md.attn_R;
      // Query tiles per work item (a row's result does not depend on it):
      // one, or every tile of a KV head's queries together, up to four, one
      // team of warps each.
      {
        const int ntiles = (rs.rps * (c.n_heads / c.n_kv_heads) + 15) / 16;
        t.TG = !md.attn_group ? 1 : (ntiles >= 3 ? 4 : ntiles);
      }
      t.stages = md.attn_stages;
      t.q = e->q;
      t.part = e->apart;
      t.out = e->fo;
      t.nq = c.n_heads;
      t.nkv = c.n_kv_heads;
      t.hd = c.head_dim;
      t.s_max = e->s_max;
      t.B = seq >= 0 ? 1 : e->B;
      t.n_kv_chunks = e->lay.n_kv_chunks;
      t.scale = 1.0f / sqrtf((float)c.head_dim);
      t.err = e->st.err;
      t.umma = tc;
      t.rs = traced(e, rs, "attention");
      t.merge_trace_id = traced(e, rs, "merge").trace_id;
      CK(launch_attention(t, e->num_sms, s, e->pdl));
      // o-projection + residual
      a = base_args(e, md, tc ? md.u_o : md.p_o, rs);
      a.w[0] = lw.w[W_O];
      maps(a, lw, 0, W_O);
      a.nf4 = nf4;
      a.stages = stages(a);
      uplan_args(a, tc ? md.u_o : md.p_o);
      a.seg_end[0] = H;
      a.ld[0] = QD;
      a.nseg = 1;
      a.N = H;
      a.K = QD;
      a.in = reinterpret_cast<const uint4*>(e->fo);
      a.out = e->x;
      a.out_ld = H;
      a.ssq_out = e->ssq;
      a.frag_out = e->fh;
      a.frag_gain = lw.ln2;
      a.frag_umma = tc;
      a.rs = traced(e, rs, "o_proj");
      CK(gemm(a, EPI_RESID));
      // gate/up + SwiGLU
      a = base_args(e, md, tc ? md.u_gu : md.p_gu, rs);
      a.w[0] = lw.w[W_G];
      a.w[1] = lw.w[W_U];
      maps(a, lw, 0, W_G);
      maps(a, lw, 1, W_U);
      a.nf4 = nf4;
      a.stages = stages(a);
      uplan_args(a, tc ? md.u_gu : md.p_gu);
      a.ld[0] = a.ld[1] = H;
      a.nseg = 2;
      a.N = c.ffn;
      a.K = H;
      a.in = reinterpret_cast<const uint4*>(e->fh);
      a.ssq = e->ssq;
      a.nssq = H / 128;
      a.inv_k = 1.0f / H;
      a.frag_out = e->fa;
      a.frag_umma = tc;
      a.rs = traced(e, rs, "gate_up");
      CK(gemm(a, EPI_SWIGLU));
      // down + residual
      a = base_args(e, md, tc ? md.u_d : md.p_d, rs);
      a.w[0] = lw.w[W_D];
      maps(a, lw, 0, W_D);
      a.nf4 = nf4;
      a.stages = stages(a);
      uplan_args(a, tc ? md.u_d : md.p_d);
      a.seg_end[0] = H;
      a.ld[0] = c.ffn;
      a.nseg = 1;
      a.N = H;
      a.K = c.ffn;
      a.in = reinterpret_cast<const uint4*>(e->fa);
      a.out = e->x;
      a.out_ld = H;
      a.ssq_out = e->ssq;
      a.frag_out = e->fx;   // the next layer's QKV input, or the LM head's
      a.frag_gain = l + 1 < c.layers ? md.L[l + 1].ln1 : md.norm;
      a.frag_umma = tc;   // the next layer's QKV or the LM head, same kernel family
      a.rs = traced(e, rs, "down");
      CK(gemm(a, EPI_RESID));
    }
  }
  if (!lm) return SF_OK;
  GemmArgs a = base_args(e, md, tc ? md.u_lm : md.p_lm, rs);
  a.w[0] = md.lm;
  a.tm[0] = tc ? md.lm_tmu : md.lm_tm;
  a.seg_end[0] = c.vocab;
  a.ld[0] = md.lm_ld;
  a.nseg = 1;
  a.N = c.vocab;
  a.K = H;
  a.in = reinterpret_cast<const uint4*>(e->fx);
  a.ssq = e->ssq;
  a.nssq = H / 128;
  a.inv_k = 1.0f / H;
  a.keys = e->keys;
  a.done = e->done;
  a.tok_out = to.tok;
  a.tok_stride = to.stride;
  a.tok_skip = to.skip;
  a.tok_off = to.off;
  a.logits = to.logits;
  a.lg_stride = to.lg_stride;
  a.lg_off = to.lg_off;
  a.rs = traced(e, rs, "lm_head");
  if (f32) {
    CK(launch_gemm_f32(a, EPI_ARGMAX, s, e->pdl));
  } else if (tc) {
    a.stages = umma_stages(rs.M, false);
    CK(launch_umma(a, EPI_ARGMAX, s, e->pdl));
  } else {
    a.stages = 5;
    CK(launch_lmhead(a, e->num_sms, s, e->pdl));
  }
  return SF_OK;
}

sf_status enqueue_draft(sf_engine* e, float* logits, cudaStream_t s) {
  const int K1 = e->K + 1;
  // Step 0: rows (committed[C-2], committed[C-1]) at positions C-2, C-1.
  RowSet rs{e->st.dtok0, 2, 0, 2, 2 * e->B, e->st.len_d, 0};
  TokOut to;
  to.tok = e->st.vtok;
  to.stride = K1;
  to.skip = 1;
  to.off = 1;
  to.logits = logits;
  to.lg_stride = e->K;
  to.lg_off = 0;
  sf_status r = forward(e, e->dft, rs, true, to, s);
  if (r != SF_OK) return r;
  for (int i = 1; i < e->K; ++i) {
    // Step i: d_i at position C - 1 + i.
    RowSet ri{e->st.vtok, K1, i, 1, e->B, e->st.len_d, 1 + i};
    TokOut ti;
    ti.tok = e->st.vtok;
    ti.stride = K1;
    ti.skip = 0;
    ti.off = i + 1;
    ti.logits = logits;
    ti.lg_stride = e->K;
    ti.lg_off = i;
    if ((r = forward(e, e->dft, ri, true, ti, s)) != SF_OK) return r;
  }
  return SF_OK;
}

// tree_g > 0: the rows are candidate guesses of tree_g tokens each (see RowSet).
sf_status enqueue_verify(sf_engine* e, float* logits, cudaStream_t s, int tree_g = 0) {
  const int K1 = e->K + 1;
  RowSet rs{e->st.vtok, K1, 0, K1, e->B * K1, e->st.len_t, 0};
  rs.tree_g = tree_g;
  TokOut to;
  to.tok = e->st.ttok;
  to.stride = K1;
  to.skip = 0;
  to.off = 0;
  to.logits = logits;
  to.lg_stride = K1;
  to.lg_off = 0;
  return forward(e, e->tgt, rs, true, to, s);
}

// Acceptance over the candidates, then the winner's cache entries move down
// to the committed slots.
sf_status enqueue_tree_accept(sf_engine* e, int n_cand, cudaStream_t s, bool pdl) {
  const int g = e->K / n_cand;
  CK(launch_accept_tree(e->st, n_cand, g, s, pdl));
  const sf_model_cfg& c = e->tgt.c;
  CK(launch_tree_compact(e->st, e->tgt.kv, c.layers, c.n_kv_heads, c.head_dim, g, s, pdl));
  return SF_OK;
}

// One round with several prompt-lookup guesses verified side by side.
sf_status enqueue_tree_round(sf_engine* e, int n_cand, int min_n, int max_n, cudaStream_t s) {
  const int g = e->K / n_cand;
  CK(launch_ngram_tree(e->st, n_cand, g, min_n, max_n, nullptr, nullptr, s, e->pdl));
  sf_status r = enqueue_verify(e, nullptr, s, g);
  if (r != SF_OK) return r;
  return enqueue_tree_accept(e, n_cand, s, e->pdl);
}

sf_status enqueue_round(sf_engine* e, int mode, cudaStream_t s) {
  sf_status r;
  if (mode == SF_DRAFT_NEURAL) {
    if ((r = enqueue_draft(e, nullptr, s)) != SF_OK) return r;
  } else if (mode == SF_DRAFT_NGRAM) {
    CK(launch_ngram(e->st, e->K, e->ng_min, e->ng_max, nullptr, nullptr, s, e->pdl));
  } else if (mode == SF_DRAFT_TREE) {
    return enqueue_tree_round(e, e->tree_n, e->ng_min, e->ng_max, s);
  } else {
    // No drafter: the lookup kernel with an empty range of n proposes nothing,
    // so the round commits the target's own next token (plain greedy decoding).
    CK(launch_ngram(e->st, e->K, 1, 0, nullptr, nullptr, s, e->pdl));
  }
  if ((r = enqueue_verify(e, nullptr, s)) != SF_OK) return r;
  CK(launch_accept(e->st, mode, s, e->pdl));
  return SF_OK;
}

enum {
  CAP_ROUND_NEURAL = 0, CAP_ROUND_NGRAM = 1, CAP_ROUND_NONE = 2, CAP_ROUND_TREE = 3,
  CAP_DRAFT = 4, CAP_VERIFY = 5, CAP_VERIFY_TREE = 6
};

cudaGraphExec_t* graph_slot(sf_engine* e, int what) {
  if (what == CAP_DRAFT) return &e->g_draft;
  if (what == CAP_VERIFY) return &e->g_verify;
  if (what == CAP_VERIFY_TREE) return &e->g_verify_tree;
  return &e->graph[what];
}

// Capture (once) the launches of `what` on the private stream and keep the
// instantiated graph; replays then cost one launch.
sf_status build_graph(sf_engine* e, int what) {
  cudaGraphExec_t* slot = graph_slot(e, what);
  if (*slot) return SF_OK;
  CK(cudaStreamBeginCapture(e->cap, cudaStreamCaptureModeThreadLocal));
  sf_status r;
  if (what == CAP_DRAFT) r = enqueue_draft(e, nullptr, e->cap);
  else if (what == CAP_VERIFY) r = enqueue_verify(e, nullptr, e->cap);
  else if (what == CAP_VERIFY_TREE) r = enqueue_verify(e, nullptr, e->cap, e->K / e->drafted_tree_n);
  else r = enqueue_round(e, what, e->cap);
  cudaGraph_t g = nullptr;
  cudaError_t ce = cudaStreamEndCapture(e->cap, &g);
  if (r != SF_OK) {
    if (g) cudaGraphDestroy(g);
    return r;
  }
  if (ce != cudaSuccess) return fail(SF_ERR_CUDA, "graph capture failed: %s", cudaGetErrorString(ce));
  if (what <= CAP_ROUND_TREE) {
    size_t n = 0;
    if (cudaGraphGetNodes(g, nullptr, &n) == cudaSuccess) e->graph_kernels[what] = n;
  }
  ce = cudaGraphInstantiate(slot, g, 0);
  cudaGraphDestroy(g);
  if (what == CAP_VERIFY_TREE && ce == cudaSuccess) e->g_verify_tree_g = e->K / e->drafted_tree_n;
  if (ce != cudaSuccess) return fail(SF_ERR_CUDA, "graph instantiate failed: %s", cudaGetErrorString(ce));
  return SF_OK;
}

// The whole generation as one graph: a WHILE conditional node whose body is
// the round of drafter `mode` followed by the loop control kernel (see
// k_loop_ctl), captured into the body with the kernels' programmatic
// dependent launches; if the body does not take them, it is captured without.
sf_status build_loop_graph(sf_engine* e, int mode) {
  if (e->loop[mode]) return SF_OK;
  cudaError_t last = cudaSuccess;
  for (int attempt = 0; attempt < 2; ++attempt) {
    const bool pdl_saved = e->pdl;
    if (attempt == 1) e->pdl = false;
    cudaGraph_t g = nullptr;
    cudaGraphExec_t ex = nullptr;
    size_t nodes = 0;
    sf_status r = SF_OK;
    cudaError_t ce = cudaGraphCreate(&g, 0);
    cudaGraphConditionalHandle hnd{};
    if (ce == cudaSuccess) ce = cudaGraphConditionalHandleCreate(&hnd, g, 1, cudaGraphCondAssignDefault);
    cudaGraph_t body = nullptr;
    if (ce == cudaSuccess) {
      cudaGraphNodeParams np = {};
      np.type = cudaGraphNodeTypeConditional;
      np.conditional.handle = hnd;
      np.conditional.type = cudaGraphCondTypeWhile;
      np.conditional.size = 1;
      cudaGraphNode_t node;
      ce = cudaGraphAddNode(&node, g, nullptr, nullptr, 0, &np);
      if (ce == cudaSuccess) body = np.conditional.phGraph_out[0];
    }
    if (ce == cudaSuccess) ce = cudaStreamBeginCaptureToGraph(e->cap, body, nullptr, nullptr, 0,
                                                              cudaStreamCaptureModeThreadLocal);
    if (ce == cudaSuccess) {
      r = enqueue_round(e, mode, e->cap);
      const cudaError_t lc = r == SF_OK ? launch_loop_ctl(e->st, hnd, e->cap) : cudaSuccess;
      cudaGraph_t out = nullptr;
      ce = cudaStreamEndCapture(e->cap, &out);
      if (ce == cudaSuccess) ce = lc;
    }
    if (ce == cudaSuccess && r == SF_OK) {
      cudaGraphGetNodes(body, nullptr, &nodes);
      ce = cudaGraphInstantiate(&ex, g, 0);
    }
    e->pdl = pdl_saved;
    if (g) cudaGraphDestroy(g);
    if (r != SF_OK) return r;
    if (ce == cudaSuccess) {
      e->loop[mode] = ex;
      if (!e->graph_kernels[mode] && nodes > 0) e->graph_kernels[mode] = nodes - 1;   // the round without the control kernel
      return SF_OK;
    }
    cudaGetLastError();   // clear a sticky launch error of the failed attempt
    last = ce;
  }
  return fail(SF_ERR_CUDA, "device loop graph: %s", cudaGetErrorString(last));
}

// The persistent decode forward for model `md`: shapes it handles (bf16
// weights; H a multiple of 128 for the LM head's sums of squares; every row
// of 16-byte pieces; at most 16 query rows of a KV head over two token rows
// and 2048 (row, dimension) outputs per attention item), the most rows whose
// shared memory fits in kDecSmemMax, and the device table of its layer pointers.
constexpr int kDecSmemMax = 200 * 1024;

int decode_smem(const sf_engine* e, const Model& md, int rows) {
  const sf_model_cfg& c = md.c;
  return decode_smem_bytes(rows, c.hidden, c.n_heads * c.head_dim, c.ffn, c.head_dim, c.n_heads / c.n_kv_heads, 2,
                           e->lay.n_kv_chunks);
}

sf_status setup_decode(sf_engine* e, Model& md, DecLayer* dev, int* smem_need) {
  const sf_model_cfg& c = md.c;
  const int group = c.n_heads / c.n_kv_heads;
  int rows = 4;
  while (rows > 0 && decode_smem(e, md, rows) > kDecSmemMax) --rows;
  if (!e->dec_on || rows == 0 || c.wdtype != SF_WDTYPE_BF16 || c.hidden % 128 || c.ffn % 8 || c.head_dim % 8 ||
      md.embed_ld % 8 || 2 * group > 16 || 2 * group * c.head_dim > 2048 || c.n_kv_heads > 64)
    return SF_OK;
  const int smem = decode_smem(e, md, rows);
  std::vector<DecLayer> t(c.layers);
  for (int l = 0; l < c.layers; ++l) {
    const LayerW& lw = md.L[l];
    auto b = [](const void* p) { return static_cast<const bf16*>(p); };
    t[l] = DecLayer{b(lw.ln1), b(lw.w[W_Q]), b(lw.w[W_K]), b(lw.w[W_V]), b(lw.bq), b(lw.bk), b(lw.bv),
                    b(lw.w[W_O]), b(lw.ln2), b(lw.w[W_G]), b(lw.w[W_U]), b(lw.w[W_D])};
  }
  CK(cudaMemcpyAsync(dev, t.data(), t.size() * sizeof(DecLayer), cudaMemcpyHostToDevice, e->user));
  CK(cudaStreamSynchronize(e->user));
  md.dlay = dev;
  md.dec_rows = rows;
  *smem_need = std::max(*smem_need, smem);
  return SF_OK;
}

// Copy the report block to pinned memory, wait, and turn device error bits
// into a status (clearing them).
sf_status sync_report(sf_engine* e) {
  CK(cudaMemcpyAsync(e->pin, e->st.ncommit, e->so.report_ints * sizeof(int), cudaMemcpyDeviceToHost, e->user));
  CK(cudaStreamSynchronize(e->user));
  const int err = e->pin[e->so.err - e->so.report];
  if (err) {
    CK(cudaMemsetAsync(e->st.err, 0, sizeof(int), e->user));
    // A barrier wait that gave up leaves the persistent kernel's barrier
    // words inconsistent: start them afresh (no kernel is running now).
    if (err & kErrWait) CK(cudaMemsetAsync(e->dbar, 0, 16 + 4 * 64 * 4, e->user));
    CK(cudaStreamSynchronize(e->user));
    if (err & kErrWait) return fail(SF_ERR_DEVICE, "a kernel's bounded wait expired (device flag %d)", err);
    if (err & kErrNonfinite) return fail(SF_ERR_NONFINITE, "non-finite logits (device flag %d)", err);
    return fail(SF_ERR_CAPACITY, "cache capacity or token range exceeded on the device (flag %d)", err);
  }
  const int* tot = e->pin + (e->so.total - e->so.report);
  for (int b = 0; b < e->B; ++b) e->C[b] = e->P[b] + tot[b];
  return SF_OK;
}

int max_committed(const sf_engine* e) {
  int m = 0;
  for (int v : e->C) m = std::max(m, v);
  return m;
}

}  // namespace

// =================================================================== C ABI
extern "C" {

int32_t sf_weight_count(const sf_model_cfg* cfg) {
  if (!cfg || cfg->layers < 1) return -1;
  if (cfg->wdtype < SF_WDTYPE_BF16 || cfg->wdtype > SF_WDTYPE_F32) return -1;
  const int per_layer = cfg->wdtype == SF_WDTYPE_NF4 ? 12 + 7 : 12;
  return 1 + cfg->layers * per_layer + 1 + (cfg->tied ? 0 : 1);
}

size_t sf_kv_bytes(const sf_model_cfg* cfg, int32_t batch, int32_t s_max) {
  if (!cfg || batch < 1 || s_max < 1) return 0;
  return (size_t)cfg->layers * 2 * batch * cfg->n_kv_heads * (size_t)s_max * cfg->head_dim * 2;
}

size_t sf_workspace_bytes(const sf_model_cfg* tgt, const sf_model_cfg* dft, int32_t batch, int32_t K,
                          int32_t s_max) {
  std::string why;
  if (!cfg_ok(tgt, &why) || (dft && !cfg_ok(dft, &why)) || batch < 1 || K < 1 || s_max < 64 ||
      s_max % kKvChunk)
    return 0;
  return make_layout(tgt, dft, batch, K, s_max).total;
}

const char* sf_status_str(sf_status s) {
  switch (s) {
    case SF_OK: return "ok";
    case SF_ERR_ARG: return "invalid argument";
    case SF_ERR_CAPACITY: return "cache capacity exceeded";
    case SF_ERR_CUDA: return "CUDA error";
    case SF_ERR_NONFINITE: return "non-finite logits";
    case SF_ERR_STATE: return "call out of order";
    case SF_ERR_UNSUPPORTED: return "unsupported shape or mode";
    case SF_ERR_DEVICE: return "device-side wait expired";
    default: return "unknown status";
  }
}

const char* sf_last_error(void) { return g_err.c_str(); }

sf_status sf_create(const sf_model_cfg* tgt, const void* const* tgt_w, const sf_model_cfg* dft,
                    const void* const* dft_w, int32_t batch, int32_t K, int32_t s_max, void* kv_t, void* kv_d,
                    void* workspace, void* cuda_stream, sf_handle* out) {
  if (!out) return fail(SF_ERR_ARG, "out is null");
  *out = nullptr;
  std::string why;
  if (!cfg_ok(tgt, &why)) return fail(SF_ERR_ARG, "target: %s", why.c_str());
  if (dft && !cfg_ok(dft, &why)) return fail(SF_ERR_ARG, "draft: %s", why.c_str());
  if (!tgt_w || (dft && !dft_w)) return fail(SF_ERR_ARG, "weight pointer array is null");
  if (batch < 1 || batch > 32 || K < 1 || K > 15) return fail(SF_ERR_ARG, "need batch in 1..32 and K in 1..15");
  if (batch * (K + 1) > SF_MAX_ROWS || batch * 2 > SF_MAX_ROWS)
    return fail(SF_ERR_UNSUPPORTED, "batch*(K+1) = %d exceeds %d rows", batch * (K + 1), SF_MAX_ROWS);
  if (s_max < 64 || s_max % kKvChunk || s_max > 16384)
    return fail(SF_ERR_ARG, "s_max must be a multiple of 64 in 64..16384");
  if (!kv_t || (dft && !kv_d) || !workspace) return fail(SF_ERR_ARG, "null cache or workspace pointer");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) || (reinterpret_cast<uintptr_t>(kv_t) & 255) ||
      (kv_d && (reinterpret_cast<uintptr_t>(kv_d) & 255)))
    return fail(SF_ERR_ARG, "workspace and caches must be 256-byte aligned");
  if (dft && dft->vocab != tgt->vocab)
    return fail(SF_ERR_ARG, "draft and target vocabularies differ (%d vs %d)", dft->vocab, tgt->vocab);

  sf_engine* e = new sf_engine();
  e->B = batch;
  e->K = K;
  e->s_max = s_max;
  e->user = static_cast<cudaStream_t>(cuda_stream);
  e->has_dft = dft != nullptr;
  e->drafter = dft ? SF_DRAFT_NEURAL : SF_DRAFT_NGRAM;
  e->tree_n = K >= 2 ? 2 : 1;
  // SF_PDL=0 in the environment launches the kernels without programmatic
  // dependent launch (for comparing the two; results are identical).
  if (const char* v = getenv("SF_PDL")) e->pdl = v[0] != '0';
  // SF_PERSISTENT=1: forwards of at most four rows run as the persistent
  // decode kernel instead of the per-projection kernels (measured slower on
  // GB300 for the draft step: it is kept as an alternative, not the default).
  if (const char* v = getenv("SF_PERSISTENT")) e->dec_on = v[0] == '1';
  // SF_KV_BOX8=1: the attention kernel loads a sequence's partly filled last
  // cache chunk in 8-slot boxes instead of whole (results are identical;
  // measured slightly slower on GB300, so off by default).
  if (const char* v = getenv("SF_KV_BOX8")) e->box8 = v[0] == '1';
  // SF_TEST_WAIT_EXPIRE=1: the first weight-tile wait of every projection
  // gives up at once and reports it (the wait then completes normally), so
  // tests can drive the device error path without stalling a kernel.
  if (const char* v = getenv("SF_TEST_WAIT_EXPIRE")) e->expire_waits = v[0] == '1';
  // SF_HOST_LOOP=1: sf_generate replays the round graph from the host (for
  // comparing with the device-resident loop; results are identical).
  if (const char* v = getenv("SF_HOST_LOOP")) e->host_loop = v[0] == '1';
  // SF_TRACE=1: kernels stamp a launch timeline (see sf_trace).
  const char* tr = getenv("SF_TRACE");
  const bool trace_on = tr && tr[0] == '1';
  auto bail = [&](sf_status s) {
    sf_destroy(e);
    return s;
  };
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&e->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return bail(fail(SF_ERR_CUDA, "no CUDA device"));
  e->slots = 2 * e->num_sms;
  {
    const cudaError_t ge = gemm_init();   // before planning: cluster occupancy queries need it
    if (ge != cudaSuccess) return bail(fail(SF_ERR_CUDA, "gemm_init: %s", cudaGetErrorString(ge)));
  }
  sf_status r = bind_model(e, e->tgt, tgt, tgt_w, static_cast<bf16*>(kv_t));
  if (r != SF_OK) return bail(r);
  if (dft && (r = bind_model(e, e->dft, dft, dft_w, static_cast<bf16*>(kv_d))) != SF_OK) return bail(r);

  e->lay = make_layout(tgt, dft, batch, K, s_max);
  e->so = state_offsets(batch, K, s_max);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  e->ws = ws;
  e->x = reinterpret_cast<float*>(ws + e->lay.x);
  e->ssq = reinterpret_cast<float*>(ws + e->lay.ssq);
  e->q = reinterpret_cast<float*>(ws + e->lay.q);
  e->fx = reinterpret_cast<bf16*>(ws + e->lay.fx);
  e->fh = reinterpret_cast<bf16*>(ws + e->lay.fh);
  e->fo = reinterpret_cast<bf16*>(ws + e->lay.fo);
  e->fa = reinterpret_cast<bf16*>(ws + e->lay.fa);
  e->apart = reinterpret_cast<float*>(ws + e->lay.apart);
  e->upart = reinterpret_cast<float*>(ws + e->lay.upart);
  e->counters = reinterpret_cast<int*>(ws + e->lay.counters);
  e->keys = reinterpret_cast<unsigned long long*>(ws + e->lay.keys);
  e->done = reinterpret_cast<int*>(ws + e->lay.done);
  e->zeros = reinterpret_cast<int*>(ws + e->lay.zeros);
  e->tgt.rope = reinterpret_cast<float2*>(ws + e->lay.rope_t);
  e->dh = reinterpret_cast<float*>(ws + e->lay.dh);
  e->dbar = reinterpret_cast<unsigned*>(ws + e->lay.dbar);
  if (trace_on) e->trace = reinterpret_cast<unsigned long long*>(ws + e->lay.trace);
  if (dft) e->dft.rope = reinterpret_cast<float2*>(ws + e->lay.rope_d);
  int* S = reinterpret_cast<int*>(ws + e->lay.state);
  SpecState& st = e->st;
  st.len_t = S + e->so.len_t;
  st.len_d = S + e->so.len_d;
  st.vtok = S + e->so.vtok;
  st.ttok = S + e->so.ttok;
  st.dtok0 = S + e->so.dtok0;
  st.nprop = S + e->so.nprop;
  st.hist = S + e->so.hist;
  st.prompt_len = S + e->so.prompt_len;
  st.acc_hist = S + e->so.acc_hist;
  st.ncommit = S + e->so.ncommit;
  st.nacc = S + e->so.nacc;
  st.commit = S + e->so.commit;
  st.total = S + e->so.total;
  st.err = S + e->so.err;
  st.loop_target = S + e->so.loop_target;
  st.rounds = S + e->so.rounds;
  st.clen = S + e->so.clen;
  st.tree_c = S + e->so.tree_c;
  st.B = batch;
  st.K = K;
  st.s_max = s_max;
  e->C.assign(batch, 0);

  cudaError_t ce;
  if ((ce = attn_init()) != cudaSuccess) return bail(fail(SF_ERR_CUDA, "attn_init: %s", cudaGetErrorString(ce)));
  if (tgt->wdtype == SF_WDTYPE_NF4 || (dft && dft->wdtype == SF_WDTYPE_NF4)) {
    double lv[16];
    float lf[16];
    nf4_levels(lv);
    for (int k = 0; k < 16; ++k) lf[k] = (float)lv[k];
    if ((ce = set_nf4_levels(lf)) != cudaSuccess || (ce = set_umma_nf4_levels(lf)) != cudaSuccess)
      return bail(fail(SF_ERR_CUDA, "NF4 levels: %s", cudaGetErrorString(ce)));
  }
  // Zero everything that must start at zero: counters, keys, state.
  if ((ce = cudaMemsetAsync(ws + e->lay.counters, 0, e->lay.rope_t - e->lay.counters, e->user)) ||
      (ce = cudaMemsetAsync(ws + e->lay.state, 0, e->so.n_ints * 4, e->user)) ||
      (ce = launch_rope_table(e->tgt.rope, s_max, tgt->head_dim, tgt->rope_theta, e->user)) ||
      (dft && (ce = launch_rope_table(e->dft.rope, s_max, dft->head_dim, dft->rope_theta, e->user))) ||
      (ce = cudaStreamCreateWithFlags(&e->cap, cudaStreamNonBlocking)) ||
      (ce = cudaHostAlloc(reinterpret_cast<void**>(&e->pin), e->so.report_ints * sizeof(int) + 64,
                          cudaHostAllocDefault)) ||
      (ce = cudaMemsetAsync(e->dbar, 0, 16 + 4 * 64 * 4, e->user)) ||
      (ce = cudaStreamSynchronize(e->user)))
    return bail(fail(SF_ERR_CUDA, "sf_create set-up: %s", cudaGetErrorString(ce)));
  {
    int smem = 0;
    sf_status dr = setup_decode(e, e->tgt, reinterpret_cast<DecLayer*>(ws + e->lay.dlay_t), &smem);
    if (dr == SF_OK && dft) dr = setup_decode(e, e->dft, reinterpret_cast<DecLayer*>(ws + e->lay.dlay_d), &smem);
    if (dr != SF_OK) return bail(dr);
    if (smem > 0 && (ce = decode_init(smem)) != cudaSuccess)
      return bail(fail(SF_ERR_CUDA, "decode_init: %s", cudaGetErrorString(ce)));
  }
  *out = e;
  return SF_OK;
}

void sf_destroy(sf_handle h) {
  if (!h) return;
  for (auto& g : h->graph)
    if (g) cudaGraphExecDestroy(g);
  for (auto& g : h->loop)
    if (g) cudaGraphExecDestroy(g);
  if (h->g_draft) cudaGraphExecDestroy(h->g_draft);
  if (h->g_verify) cudaGraphExecDestroy(h->g_verify);
  if (h->g_verify_tree) cudaGraphExecDestroy(h->g_verify_tree);
  if (h->cap) cudaStreamDestroy(h->cap);
  if (h->pin) cudaFreeHost(h->pin);
  delete h;
}

sf_status sf_prefill(sf_handle h, const int32_t* h_tokens, const int32_t* h_lens, int32_t stride) {
  if (!h || !h_tokens || !h_lens) return fail(SF_ERR_ARG, "null argument");
  std::vector<int> lens(h_lens, h_lens + h->B);
  bool equal = true;
  for (int b = 0; b < h->B; ++b) {
    const int P = lens[b];
    if (P < 2 || stride < P) return fail(SF_ERR_ARG, "prompt %d: length must be >= 2 and <= stride", b);
    if (P + h->K + 1 > h->s_max)
      return fail(SF_ERR_CAPACITY, "prompt %d of %d tokens leaves no room for a round", b, P);
    for (int i = 0; i < P; ++i) {
      const int t = h_tokens[(size_t)b * stride + i];
      if (t < 0 || t >= h->tgt.c.vocab) return fail(SF_ERR_ARG, "token %d out of range at [%d][%d]", t, b, i);
    }
    equal = equal && P == lens[0];
  }
  for (int b = 0; b < h->B; ++b)
    CK(cudaMemcpyAsync(h->st.hist + (size_t)b * h->s_max, h_tokens + (size_t)b * stride, lens[b] * sizeof(int),
                       cudaMemcpyHostToDevice, h->user));
  CK(cudaMemcpyAsync(h->st.prompt_len, lens.data(), h->B * sizeof(int), cudaMemcpyHostToDevice, h->user));
  CK(launch_reset(h->st, h->user));
  // Fill the caches with prompt[0..P-1) in chunks of up to SF_MAX_ROWS rows:
  // all sequences side by side when the prompts have one length, else one
  // sequence at a time.
  for (Model* md : {&h->tgt, &h->dft}) {
    if (md == &h->dft && !h->has_dft) continue;
    if (equal) {
      const int P = lens[0], cl = SF_MAX_ROWS / h->B;
      for (int start = 0; start < P - 1; start += cl) {
        const int n = std::min(cl, P - 1 - start);
        RowSet rs{h->st.hist, h->s_max, start, n, h->B * n, h->zeros, start};
        sf_status r = forward(h, *md, rs, false, TokOut(), h->user);
        if (r != SF_OK) return r;
      }
      continue;
    }
    for (int b = 0; b < h->B; ++b)
      for (int start = 0; start < lens[b] - 1; start += SF_MAX_ROWS) {
        const int n = std::min(SF_MAX_ROWS, lens[b] - 1 - start);
        RowSet rs{h->st.hist + (size_t)b * h->s_max, h->s_max, start, n, n, h->zeros, start};
        sf_status r = forward(h, *md, rs, false, TokOut(), h->user, b);
        if (r != SF_OK) return r;
      }
  }
  CK(cudaStreamSynchronize(h->user));
  h->P = lens;
  h->C = lens;
  h->phase = 1;
  h->draft_stale = false;
  return SF_OK;
}

sf_status sf_reset(sf_handle h) {
  if (!h) return fail(SF_ERR_ARG, "null handle");
  if (h->phase == 0) return fail(SF_ERR_STATE, "no prompt loaded");
  CK(launch_reset(h->st, h->user));
  CK(cudaStreamSynchronize(h->user));
  h->C = h->P;
  h->phase = 1;
  h->draft_stale = false;
  return SF_OK;
}

// Drop the round graphs of drafter `mode` (their launches carry its settings).
static void drop_round_graphs(sf_handle h, int mode) {
  if (h->graph[mode]) {
    cudaGraphExecDestroy(h->graph[mode]);
    h->graph[mode] = nullptr;
  }
  if (h->loop[mode]) {
    cudaGraphExecDestroy(h->loop[mode]);
    h->loop[mode] = nullptr;
  }
  h->graph_kernels[mode] = 0;
}

sf_status sf_set_drafter(sf_handle h, int32_t mode, int32_t min_n, int32_t max_n) {
  if (!h) return fail(SF_ERR_ARG, "null handle");
  if (mode != SF_DRAFT_NEURAL && mode != SF_DRAFT_NGRAM && mode != SF_DRAFT_NONE && mode != SF_DRAFT_TREE)
    return fail(SF_ERR_ARG, "unknown drafter");
  if (mode == SF_DRAFT_NEURAL && !h->has_dft) return fail(SF_ERR_STATE, "no draft model");
  const bool lookup = mode == SF_DRAFT_NGRAM || mode == SF_DRAFT_TREE;
  if (lookup && (min_n < 1 || max_n < min_n || max_n > 64)) return fail(SF_ERR_ARG, "need 1 <= min_n <= max_n <= 64");
  if (lookup && (min_n != h->ng_min || max_n != h->ng_max)) {
    drop_round_graphs(h, SF_DRAFT_NGRAM);
    drop_round_graphs(h, SF_DRAFT_TREE);
    h->ng_min = min_n;
    h->ng_max = max_n;
  }
  h->drafter = mode;
  return SF_OK;
}

sf_status sf_set_tree_candidates(sf_handle h, int32_t n_cand) {
  if (!h) return fail(SF_ERR_ARG, "null handle");
  if (n_cand < 1 || n_cand > h->K) return fail(SF_ERR_ARG, "need 1 <= n_cand <= K");
  if (n_cand != h->tree_n) {
    drop_round_graphs(h, SF_DRAFT_TREE);
    h->tree_n = n_cand;
  }
  return SF_OK;
}

sf_status sf_draft(sf_handle h, int32_t* d_draft, float* d_logits) {
  if (!h) return fail(SF_ERR_ARG, "null handle");
  if (!h->has_dft) return fail(SF_ERR_STATE, "no draft model");
  if (h->phase != 1) return fail(SF_ERR_STATE, "sf_draft needs a prefilled engine between rounds");
  if (h->draft_stale) return fail(SF_ERR_STATE, "draft cache is behind after n-gram rounds; call sf_reset or sf_prefill");
  if (max_committed(h) + h->K + 1 > h->s_max) return fail(SF_ERR_CAPACITY, "round would exceed s_max");
  sf_status r;
  if (!d_draft && !d_logits) {
    if ((r = build_graph(h, CAP_DRAFT)) != SF_OK) return r;
    CK(cudaGraphLaunch(h->g_draft, h->user));
  } else if ((r = enqueue_draft(h, d_logits, h->user)) != SF_OK) {
    return r;
  }
  if (d_draft) CK(launch_copy_draft(h->st, d_draft, h->user));
  h->phase = 2;
  h->drafted_mode = SF_DRAFT_NEURAL;
  return SF_OK;
}

sf_status sf_ngram_draft(sf_handle h, int32_t max_guess, int32_t min_n, int32_t max_n, int32_t* d_prop,
                         int32_t* d_count) {
  if (!h) return fail(SF_ERR_ARG, "null handle");
  if (h->phase != 1) return fail(SF_ERR_STATE, "sf_ngram_draft needs a prefilled engine between rounds");
  if (max_guess < 1 || max_guess > h->K || min_n < 1 || max_n < min_n || max_n > 64)
    return fail(SF_ERR_ARG, "need 1 <= max_guess <= K and 1 <= min_n <= max_n <= 64");
  if (max_committed(h) + h->K + 1 > h->s_max) return fail(SF_ERR_CAPACITY, "round would exceed s_max");
  CK(launch_ngram(h->st, max_guess, min_n, max_n, d_prop, d_count, h->user, false));
  h->phase = 2;
  h->drafted_mode = SF_DRAFT_NGRAM;
  return SF_OK;
}

sf_status sf_tree_draft(sf_handle h, int32_t n_cand, int32_t min_n, int32_t max_n, int32_t* d_prop,
                        int32_t* d_len) {
  if (!h) return fail(SF_ERR_ARG, "null handle");
  if (h->phase != 1) return fail(SF_ERR_STATE, "sf_tree_draft needs a prefilled engine between rounds");
  if (n_cand < 1 || n_cand > h->K || min_n < 1 || max_n < min_n || max_n > 64)
    return fail(SF_ERR_ARG, "need 1 <= n_cand <= K and 1 <= min_n <= max_n <= 64");
  if (max_committed(h) + h->K + 1 > h->s_max) return fail(SF_ERR_CAPACITY, "round would exceed s_max");
  CK(launch_ngram_tree(h->st, n_cand, h->K / n_cand, min_n, max_n, d_prop, d_len, h->user, false));
  h->phase = 2;
  h->drafted_mode = SF_DRAFT_TREE;
  h->drafted_tree_n = n_cand;
  return SF_OK;
}

sf_status sf_verify(sf_handle h, int32_t* d_tgt_argmax, float* d_logits) {
  if (!h) return fail(SF_ERR_ARG, "null handle");
  if (h->phase != 2) return fail(SF_ERR_STATE, "sf_verify needs a draft first");
  sf_status r;
  const bool tree = h->drafted_mode == SF_DRAFT_TREE;
  const int tree_g = tree ? h->K / h->drafted_tree_n : 0;
  if (!d_tgt_argmax && !d_logits) {
    const int what = tree ? CAP_VERIFY_TREE : CAP_VERIFY;
    if (tree && h->g_verify_tree && h->g_verify_tree_g != tree_g) {
      cudaGraphExecDestroy(h->g_verify_tree);
      h->g_verify_tree = nullptr;
    }
    if ((r = build_graph(h, what)) != SF_OK) return r;
    CK(cudaGraphLaunch(*graph_slot(h, what), h->user));
  } else if ((r = enqueue_verify(h, d_logits, h->user, tree_g)) != SF_OK) {
    return r;
  }
  if (d_tgt_argmax)
    CK(cudaMemcpyAsync(d_tgt_argmax, h->st.ttok, h->B * (h->K + 1) * sizeof(int), cudaMemcpyDeviceToDevice,
                       h->user));
  h->phase = 3;
  return SF_OK;
}

static void copy_out(sf_handle h, int32_t* h_n_accepted, int32_t* h_committed, int32_t* h_n_committed) {
  const int* rep = h->pin;
  const int K1 = h->K + 1;
  for (int b = 0; b < h->B; ++b) {
    if (h_n_committed) h_n_committed[b] = rep[h->so.ncommit - h->so.report + b];
    if (h_n_accepted) h_n_accepted[b] = rep[h->so.nacc - h->so.report + b];
    if (h_committed)
      for (int j = 0; j < K1; ++j) h_committed[b * K1 + j] = rep[h->so.commit - h->so.report + b * K1 + j];
  }
}

sf_status sf_accept_rollback(sf_handle h, int32_t* h_n_accepted, int32_t* h_committed, int32_t* h_n_committed) {
  if (!h) return fail(SF_ERR_ARG, "null handle");
  if (h->phase != 3) return fail(SF_ERR_STATE, "sf_accept_rollback needs a verify first");
  if (h->drafted_mode == SF_DRAFT_TREE) {
    const sf_status ta = enqueue_tree_accept(h, h->drafted_tree_n, h->user, false);
    if (ta != SF_OK) return ta;
  } else {
    CK(launch_accept(h->st, h->drafted_mode, h->user, false));
  }
  h->phase = 1;
  if (h->drafted_mode != SF_DRAFT_NEURAL && h->has_dft) h->draft_stale = true;
  sf_status r = sync_report(h);
  if (r != SF_OK) return r;
  copy_out(h, h_n_accepted, h_committed, h_n_committed);
  return SF_OK;
}

sf_status sf_step(sf_handle h, int32_t* h_n_committed, int32_t* h_committed) {
  if (!h) return fail(SF_ERR_ARG, "null handle");
  if (h->phase != 1) return fail(SF_ERR_STATE, "sf_step needs a prefilled engine between rounds");
  const int mode = h->drafter;
  if (mode == SF_DRAFT_NEURAL && h->draft_stale)
    return fail(SF_ERR_STATE, "draft cache is behind after n-gram rounds; call sf_reset or sf_prefill");
  if (max_committed(h) + h->K + 1 > h->s_max) return fail(SF_ERR_CAPACITY, "round would exceed s_max");
  sf_status r = build_graph(h, mode);
  if (r != SF_OK) return r;
  CK(cudaGraphLaunch(h->graph[mode], h->user));
  if (mode != SF_DRAFT_NEURAL && h->has_dft) h->draft_stale = true;
  if ((r = sync_report(h)) != SF_OK) return r;
  copy_out(h, nullptr, h_committed, h_n_committed);
  return SF_OK;
}

sf_status sf_generate(sf_handle h, int32_t n_new, int32_t* h_out, int32_t* h_rounds) {
  if (!h) return fail(SF_ERR_ARG, "null handle");
  if (h->phase != 1) return fail(SF_ERR_STATE, "sf_generate needs a prefilled engine between rounds");
  if (n_new < 1) return fail(SF_ERR_ARG, "n_new must be >= 1");
  const int mode = h->drafter;
  if (mode == SF_DRAFT_NEURAL && h->draft_stale)
    return fail(SF_ERR_STATE, "draft cache is behind after n-gram rounds; call sf_reset or sf_prefill");
  const int K1 = h->K + 1;
  auto gen_min = [&]() {
    int g = 1 << 30;
    for (int b = 0; b < h->B; ++b) g = std::min(g, h->C[b] - h->P[b]);
    return g;
  };
  int rounds = 0;
  sf_status r;
  if (!h->host_loop) {
    // Device-resident loop: one graph launch runs every round; the host
    // synchronises once at the end.
    if (gen_min() < n_new) {
      if (max_committed(h) + 2 * K1 > h->s_max) return fail(SF_ERR_CAPACITY, "s_max reached after %d new tokens", gen_min());
      if ((r = build_loop_graph(h, mode)) != SF_OK) return r;
      CK(launch_loop_init(h->st, n_new, h->user));
      CK(cudaGraphLaunch(h->loop[mode], h->user));
      if (mode != SF_DRAFT_NEURAL && h->has_dft) h->draft_stale = true;
      if ((r = sync_report(h)) != SF_OK) return r;
      rounds = h->pin[h->so.rounds - h->so.report];
      if (gen_min() < n_new) return fail(SF_ERR_CAPACITY, "s_max reached after %d new tokens", gen_min());
    }
  } else {
    if ((r = build_graph(h, mode)) != SF_OK) return r;
    for (;;) {
      const int remaining = n_new - gen_min();
      if (remaining <= 0) break;
      // Each round commits at most K+1 tokens, so this many rounds never
      // overshoots the target by more than one round's worth.
      int R = (remaining + K1 - 1) / K1;
      const int room = (h->s_max - h->K - 1 - max_committed(h)) / K1;
      R = std::min(R, room);
      if (R < 1) return fail(SF_ERR_CAPACITY, "s_max reached after %d new tokens", gen_min());
      for (int i = 0; i < R; ++i) CK(cudaGraphLaunch(h->graph[mode], h->user));
      rounds += R;
      if (mode != SF_DRAFT_NEURAL && h->has_dft) h->draft_stale = true;
      if ((r = sync_report(h)) != SF_OK) return r;
    }
  }
  if (h_out)
    for (int b = 0; b < h->B; ++b)
      CK(cudaMemcpyAsync(h_out + (size_t)b * n_new, h->st.hist + (size_t)b * h->s_max + h->P[b],
                         n_new * sizeof(int), cudaMemcpyDeviceToHost, h->user));
  CK(cudaStreamSynchronize(h->user));
  if (h_rounds) *h_rounds = rounds;
  return SF_OK;
}

sf_status sf_get_lengths(sf_handle h, int32_t* h_len_t, int32_t* h_len_d) {
  if (!h) return fail(SF_ERR_ARG, "null handle");
  if (h_len_t) CK(cudaMemcpyAsync(h_len_t, h->st.len_t, h->B * sizeof(int), cudaMemcpyDeviceToHost, h->user));
  if (h_len_d) CK(cudaMemcpyAsync(h_len_d, h->st.len_d, h->B * sizeof(int), cudaMemcpyDeviceToHost, h->user));
  CK(cudaStreamSynchronize(h->user));
  return SF_OK;
}

sf_status sf_get_accept_hist(sf_handle h, int32_t* h_hist) {
  if (!h || !h_hist) return fail(SF_ERR_ARG, "null argument");
  CK(cudaMemcpyAsync(h_hist, h->st.acc_hist, h->B * (h->K + 1) * sizeof(int), cudaMemcpyDeviceToHost, h->user));
  CK(cudaStreamSynchronize(h->user));
  return SF_OK;
}

sf_status sf_tree_winner(sf_handle h, int32_t* h_c) {
  if (!h || !h_c) return fail(SF_ERR_ARG, "null argument");
  CK(cudaMemcpyAsync(h_c, h->st.tree_c, h->B * sizeof(int), cudaMemcpyDeviceToHost, h->user));
  CK(cudaStreamSynchronize(h->user));
  return SF_OK;
}

size_t sf_linear_workspace_bytes(int32_t N, int32_t K) {
  if (N < 1 || K < 8 || K % 8) return 0;
  return align256(kLinearPartBytes) + align256((size_t)((N + 127) / 128) * kMaxGroups * 4) +
         align256(frag_bytes(K, (kRows + 3) / 4));
}

size_t sf_frag_bytes(int32_t K, int32_t M) {
  if (K < 8 || K % 8 || M < 1 || M > SF_MAX_ROWS) return 0;
  return frag_bytes(K, (M + 3) / 4);
}

sf_status sf_to_frag(const float* d_x, int32_t M, int32_t K, int32_t ld, void* d_frag, void* cuda_stream) {
  if (!d_x || !d_frag) return fail(SF_ERR_ARG, "null pointer");
  if (K < 8 || K % 8 || ld < K || M < 1 || M > SF_MAX_ROWS)
    return fail(SF_ERR_ARG, "need K a multiple of 8, ld >= K, 1 <= M <= %d", SF_MAX_ROWS);
  if (reinterpret_cast<uintptr_t>(d_frag) & 15) return fail(SF_ERR_ARG, "d_frag must be 16-byte aligned");
  CK(launch_to_frag(d_x, M, K, ld, static_cast<bf16*>(d_frag), static_cast<cudaStream_t>(cuda_stream)));
  return SF_OK;
}

sf_status sf_linear_frag(const void* d_w, int32_t N, int32_t K, int32_t ld, const void* d_frag, int32_t M,
                         float* d_y, void* d_workspace, void* cuda_stream) {
  if (!d_w || !d_frag || !d_y || !d_workspace) return fail(SF_ERR_ARG, "null pointer");
  if (N < 1 || K < 8 || K % 8 || ld < K || ld % 8 || M < 1 || M > SF_MAX_ROWS)
    return fail(SF_ERR_ARG, "need N >= 1, K and ld multiples of 8 with ld >= K, 1 <= M <= %d", SF_MAX_ROWS);
  if ((reinterpret_cast<uintptr_t>(d_w) & 15) || (reinterpret_cast<uintptr_t>(d_frag) & 15) ||
      (reinterpret_cast<uintptr_t>(d_workspace) & 255))
    return fail(SF_ERR_ARG, "W and the fragment copy must be 16-byte aligned, the workspace 256-byte aligned");
  int dev = 0, sms = 0;
  CK(cudaGetDevice(&dev));
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const bool tc = M >= umma_min_rows();   // more than 16 rows: the tcgen05 GEMM
  const Plan p = make_plan((N + 127) / 128, K, 2 * sms, tc ? 16 : 1 << 30);
  const int groups = (M + kGroupRows - 1) / kGroupRows;
  if (p.nsplit > 1 && p.nblocks * p.nsplit * groups > kLinearTiles)
    return fail(SF_ERR_UNSUPPORTED, "plan too large");
  CK(gemm_init());
  unsigned char* ws = static_cast<unsigned char*>(d_workspace);
  const size_t part_bytes = align256(kLinearPartBytes);
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (p.nsplit > 1) CK(cudaMemsetAsync(ws + part_bytes, 0, (size_t)p.nblocks * groups * 4, st));   // arrival counters
  GemmArgs a{};
  CK(make_weight_map(&a.tm[0], d_w, N, K, ld, tc ? 64 : 16));
  a.w[0] = d_w;
  a.seg_end[0] = N;
  a.ld[0] = ld;
  a.nseg = 1;
  a.N = N;
  a.K = K;
  a.nblocks = p.nblocks;
  a.nsplit = p.nsplit;
  a.cps = p.cps;
  a.stages = tc ? umma_stages(M, false) : pick_stages(p.nblocks * p.nsplit, p.cps, sms);
  a.in = static_cast<const uint4*>(d_frag);
  a.part = reinterpret_cast<float*>(ws);
  a.counter = reinterpret_cast<int*>(ws + part_bytes);
  a.out = d_y;
  a.out_ld = N;
  a.rs.M = M;
  a.rs.rps = M;
  CK(tc ? launch_umma(a, EPI_STORE, st, false) : launch_gemm(a, EPI_STORE, st, false));
  return SF_OK;
}

sf_status sf_linear(const void* d_w, int32_t N, int32_t K, int32_t ld, const float* d_x, int32_t M, float* d_y,
                    void* d_workspace, void* cuda_stream) {
  if (!d_w || !d_x || !d_y || !d_workspace) return fail(SF_ERR_ARG, "null pointer");
  if (N < 1 || K < 8 || K % 8 || ld < K || ld % 8 || M < 1 || M > SF_MAX_ROWS)
    return fail(SF_ERR_ARG, "need N >= 1, K and ld multiples of 8 with ld >= K, 1 <= M <= %d", SF_MAX_ROWS);
  if ((reinterpret_cast<uintptr_t>(d_w) & 15) || (reinterpret_cast<uintptr_t>(d_x) & 15) ||
      (reinterpret_cast<uintptr_t>(d_workspace) & 255))
    return fail(SF_ERR_ARG, "W and x must be 16-byte aligned, the workspace 256-byte aligned");
  // x -> fragment order in the workspace's last region, then the GEMM.
  unsigned char* ws = static_cast<unsigned char*>(d_workspace);
  void* xf = ws + align256(kLinearPartBytes) + align256((size_t)((N + 127) / 128) * kMaxGroups * 4);
  sf_status r = sf_to_frag(d_x, M, K, K, xf, cuda_stream);
  if (r != SF_OK) return r;
  return sf_linear_frag(d_w, N, K, ld, xf, M, d_y, d_workspace, cuda_stream);
}

int32_t sf_trace(sf_handle h, uint64_t* h_out, int32_t max_launches) {
  if (!h || !h->trace) return 0;
  if (!h_out) return h->trace_next;
  const int n = std::min(std::min(h->trace_next, kTraceSlots), max_launches);
  if (h_out && n > 0) {
    if (cudaMemcpyAsync(h_out, h->trace, (size_t)2 * n * 8, cudaMemcpyDeviceToHost, h->user) != cudaSuccess ||
        cudaStreamSynchronize(h->user) != cudaSuccess)
      return 0;
  }
  return n;
}

int64_t sf_round_launches(sf_handle h) {
  if (!h) return 0;
  return (int64_t)h->graph_kernels[h->drafter];
}

const char* sf_trace_label(sf_handle h, int32_t i) {
  if (!h || i < 0 || i >= (int)h->trace_labels.size()) return "";
  return h->trace_labels[i].c_str();
}

sf_status sf_nf4_quantize(const void* d_w, int32_t rows, int32_t cols, int32_t ld, void* d_packed, void* d_scales,
                          void* cuda_stream) {
  if (!d_w || !d_packed || !d_scales) return fail(SF_ERR_ARG, "null pointer");
  if (rows < 1 || cols < 64 || cols % 64 || ld < cols) return fail(SF_ERR_ARG, "need cols a multiple of 64 and ld >= cols");
  CK(launch_nf4_quantize(static_cast<const bf16*>(d_w), rows, cols, ld, static_cast<uint8_t*>(d_packed),
                         static_cast<__half*>(d_scales), nf4_scale_ld(cols), static_cast<cudaStream_t>(cuda_stream)));
  return SF_OK;
}

}  // extern "C"
