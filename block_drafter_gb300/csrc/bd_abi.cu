// C ABI of the drafter library: argument validation, workspace planning and the launch
// sequences of the three entry points.  Every step of the round runs in this library's
// kernels; nothing here computes on the host beyond launch geometry and the RoPE
// inverse frequencies.
#include "blockdrafter.h"
#include "bd_internal.h"
#include "bd_kernels.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>

namespace {
thread_local std::string t_last_error;

// Launch bracketing for measurement (bd_set_timing_events): while a kind is set, the
// i-th launch of that kind in a call is bracketed by begin[i] / end[i].
struct Timing {
  int kind = BD_TIME_NONE;
  int n = 0;
  int next = 0;
  cudaEvent_t begin[BD_TIMING_MAX], end[BD_TIMING_MAX];
};
thread_local Timing t_timing;
}  // namespace

namespace bd {
static std::atomic<uint64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
void set_last_error(const std::string &msg) { t_last_error = msg; }
}  // namespace bd

namespace {

using namespace bd;

bd_status fail(bd_status s, const std::string &msg) {
  t_last_error = msg;
  return s;
}

#define BD_TRY(expr)                                       \
  do {                                                     \
    std::string _e = (expr);                               \
    if (!_e.empty()) return fail(BD_ERR_CUDA, _e);         \
  } while (0)

// Records event ev on stream s; inside stream capture as an external event node of the
// graph (a plain record there would only mark a capture dependency).
std::string record_timing_event(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e == cudaSuccess)
    e = cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
                                            : cudaEventRecord(ev, s);
  return e == cudaSuccess ? std::string() : std::string("timing event: ") + cudaGetErrorString(e);
}
// Records the next begin / end event of `kind` (if that kind is being timed) on stream s.
std::string timing_begin(int kind, cudaStream_t s) {
  Timing &t = t_timing;
  if (t.kind != kind || t.next >= t.n) return {};
  return record_timing_event(t.begin[t.next], s);
}
std::string timing_end(int kind, cudaStream_t s) {
  Timing &t = t_timing;
  if (t.kind != kind || t.next >= t.n) return {};
  return record_timing_event(t.end[t.next++], s);
}
// launch_expr bracketed by the timing events of `kind`
#define BD_TIMED(kind, expr)              \
  do {                                    \
    BD_TRY(timing_begin((kind), s));      \
    BD_TRY(expr);                         \
    BD_TRY(timing_end((kind), s));        \
  } while (0)

constexpr int kMaxB = 8;
constexpr int kMaxMasks = 15;
constexpr int kMaxPendPerReq = 16;  // pending context rows a round takes per request
constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
int elem_bytes(const bd_config *c) { return c->dtype == BD_BF16 ? 2 : 4; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int sms_for_sizing() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
    return n;
  cudaGetLastError();
  return 256;  // conservative when no device is visible
}

// ------------------------------------------------------------------ validation
std::string check_config(const bd_config *c) {
  char b[256];
  if (!c) return "config is NULL";
  if (c->dtype != BD_BF16 && c->dtype != BD_F32) return "dtype must be BD_BF16 or BD_F32";
  const int e = elem_bytes(c);
  auto k_ok = [&](long long k) { return k > 0 && (k * e) % 16 == 0; };
  if (c->hidden <= 0 || !k_ok(c->hidden)) return "hidden must be > 0 and hidden*elem a multiple of 16 bytes";
  if (c->n_layers < 1 || c->n_layers > BD_MAX_LAYERS) return "n_layers out of range 1..16";
  if (c->head_dim != 64 && c->head_dim != 128) return "head_dim must be 64 or 128";
  if (c->n_kv_heads <= 0 || c->n_q_heads <= 0 || c->n_q_heads % c->n_kv_heads != 0)
    return "n_q_heads must be a positive multiple of n_kv_heads";
  if (c->ffn <= 0 || !k_ok(c->ffn)) return "ffn must be > 0 and ffn*elem a multiple of 16 bytes";
  if (c->vocab <= 0) return "vocab must be > 0";
  if (c->n_target_layers <= 0) return "n_target_layers must be > 0";
  if (c->mask_token_id < 0 || c->mask_token_id >= c->vocab) return "mask_token_id outside [0, vocab)";
  if (c->block_mask != BD_BLOCK_BIDIRECTIONAL && c->block_mask != BD_BLOCK_CAUSAL)
    return "block_mask must be 0 or 1";
  if (!(c->eps > 0.f) || !(c->rope_theta > 1.f)) return "eps must be > 0 and rope_theta > 1";
  if (c->code_width < 0 || c->msg_width < 0) return "code/message widths must be >= 0";
  if ((c->code_width > 0) != (c->msg_width > 0)) return "code_width and msg_width must both be 0 or both > 0";
  if (c->code_width > 0 && (!k_ok(c->code_width) || !k_ok(c->msg_width)))
    return "code_width*elem and msg_width*elem must be multiples of 16 bytes";
  if (c->conv_group < 0 || (c->conv_group > 0 && (c->conv_group % 4 != 0 || c->hidden % c->conv_group != 0)))
    return "conv_group must be 0 or a multiple of 4 dividing hidden";
  for (int l = 0; l < c->n_layers; ++l) {
    if (c->window[l] < 0) return "window must be >= 0";
    if (c->ring_capacity[l] <= 0) return "ring_capacity must be > 0";
    if (c->window[l] > 0 && c->ring_capacity[l] < c->window[l] - 1) {
      snprintf(b, sizeof b, "layer %d: ring_capacity %d cannot hold the %d-position window", l,
               c->ring_capacity[l], c->window[l] - 1);
      return b;
    }
  }
  return {};
}

std::string check_weights(const bd_config *c, const bd_weights *w) {
  if (!w) return "weights are NULL";
  auto chk = [](const void *p) { return p != nullptr && aligned16(p); };
  if (w->packed && (reinterpret_cast<uintptr_t>(w->packed) & 1023))
    return "packed image not 1024-byte aligned";
  if (!chk(w->w_feature) || !chk(w->context_norm) || !chk(w->final_norm) || !chk(w->embed_head))
    return "a shared weight pointer is NULL or not 16-byte aligned";
  if (c->code_width > 0) {
    if (!chk(w->codebook) || !chk(w->g_recv) || !chk(w->g_pred) || !chk(w->a_val))
      return "bridge weights (codebook, g_recv, g_pred, a_val) are NULL or misaligned";
    if (w->gate_bias && !aligned16(w->gate_bias)) return "gate_bias is not 16-byte aligned";
  }
  for (int l = 0; l < c->n_layers; ++l) {
    const bd_layer_weights &L = w->layer[l];
    if (!chk(L.in_norm) || !chk(L.wq) || !chk(L.wk) || !chk(L.wv) || !chk(L.q_norm) ||
        !chk(L.k_norm) || !chk(L.wo) || !chk(L.post_norm) || !chk(L.w_gate) || !chk(L.w_up) ||
        !chk(L.w_down))
      return "layer " + std::to_string(l) + ": a weight pointer is NULL or not 16-byte aligned";
    if (c->code_width > 0 && (!chk(L.r_read) || !chk(L.w_write)))
      return "layer " + std::to_string(l) + ": r_read / w_write NULL or misaligned";
    if (c->conv_group > 0 &&
        (!chk(L.conv_delta_a) || !chk(L.conv_base_a) || !chk(L.conv_delta_m) || !chk(L.conv_base_m)))
      return "layer " + std::to_string(l) + ": convolution weights NULL or misaligned";
  }
  return {};
}

std::string check_kv(const bd_config *c, const bd_kv_cache *kv, int B) {
  if (!kv) return "kv cache is NULL";
  if (kv->b_max < B || kv->b_max < 1) return "kv->b_max smaller than the number of requests";
  for (int l = 0; l < c->n_layers; ++l)
    if (!kv->k[l] || !kv->v[l] || !aligned16(kv->k[l]) || !aligned16(kv->v[l]))
      return "kv ring pointer NULL or misaligned";
  return {};
}

RopeFreq rope_freq(const bd_config *c) {
  RopeFreq f;
  memset(&f, 0, sizeof f);
  const int half = c->head_dim / 2;
  for (int j = 0; j < half; ++j)
    f.inv[j] = std::pow(static_cast<double>(c->rope_theta), -2.0 * j / c->head_dim);
  return f;
}

// ------------------------------------------------------------------ workspace planning
struct Carve {
  size_t off = 0;
  char *base = nullptr;
  template <typename T> T *take(size_t count) {
    T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
    off = align_up(off + count * sizeof(T));
    return p;
  }
};

// Key splits of a layer's bf16 attention (one CTA per split, KV head and request; the
// splits of a head form one cluster and merge through distributed shared memory, so the
// grid may exceed one wave): enough splits to fill the SMs once (one CTA per SM), more
// when a head's ring holds over 16 tiles of 128 slots, at most one split per tile and at
// most the portable cluster size.
int att_splits(const bd_config *c, int l, int B, int W, int sms) {
  (void)W;
  const int cap = c->ring_capacity[l];
  const int tiles = (cap + attention_tile_keys() - 1) / attention_tile_keys();
  int s = std::max(sms / (B * c->n_kv_heads), (tiles + 15) / 16);
  if (s < 1) s = 1;
  if (s > attention_max_splits()) s = attention_max_splits();
  // a grid of several waves (a long full-context window at B > 1) keeps clusters of at most
  // four: larger clusters find fewer places to run and merge more partials (measured)
  if (s > 4 && B * c->n_kv_heads * s > sms) s = 4;
  return s < tiles ? s : tiles;
}
int att_max_keys(const bd_config *c, int l, int W) {
  const int cap = c->ring_capacity[l];
  const int ctx = c->window[l] > 0 ? std::min(c->window[l] - 1, cap) : cap;
  return ctx + W;
}

// Shared scratch of every GEMM launch of one entry-point call.
struct GemmWs {
  float *partials;
  size_t partial_floats;
  unsigned *counters;
  size_t n_counters;
};
void carve_gemm(Carve &cv, GemmWs &g, int max_block_n, size_t max_tiles, int sms) {
  g.partial_floats = gemm_partial_floats(sms, max_block_n);
  g.partials = cv.take<float>(g.partial_floats);
  g.n_counters = max_tiles;
  g.counters = cv.take<unsigned>(2 * max_tiles);  // arrival and done counters
}

size_t tiles_of(int rows, int tile_rows) { return static_cast<size_t>((rows + tile_rows - 1) / tile_rows); }

struct RoundWs {
  GemmWs g;
  float *x, *z, *pre, *r, *feat, *kv_raw;
  float *cdelta_a, *cdelta_m, *cz, *cn;  // DFlash2 convolution: deltas, branch output, fp32 X
  unsigned *br_bar;    // [L][5] fused-bridge barrier counters (3 used), right after g.counters
  float *zpart, *sspart, *zsq;  // fused-bridge partial sums
  float2 *rope;
  void *xn, *xq, *cmat, *q, *kblk, *vblk, *att, *hmid, *c, *m;
};
int pad16(int n) { return (n + 15) / 16 * 16; }
// Upper bound on the n-tiles of a GEMM over n tokens.
int n_tiles_of(int n) { return gemm_max_n_tiles(n); }
// Tiles of the round's largest GEMM: the Q/K/V product also carries the T_q - T pending
// context rows, the others the T block rows; the catch-up's feature projection has H rows.
size_t round_max_tiles(const bd_config *c, int T, int Tq) {
  size_t t = (tiles_of(c->n_q_heads * c->head_dim, 128) + 2 * tiles_of(c->n_kv_heads * c->head_dim, 128)) *
             n_tiles_of(Tq);
  size_t o = std::max(tiles_of(c->hidden, 128), tiles_of(c->ffn, 64));
  if (c->code_width > 0) {
    o = std::max(o, tiles_of(c->code_width, 128));
    o = std::max(o, 3 * tiles_of(c->msg_width, 128));
  }
  if (c->conv_group > 0) t = std::max(t, tiles_of(4 * c->hidden / c->conv_group, 128) * n_tiles_of(Tq));
  return std::max(t, o * n_tiles_of(T));
}

size_t mat_max_tiles(const bd_config *c, int n);

// Pending context rows ride in the block's Q/K/V product while the product keeps a single
// n-tile (T + n_pend <= 128 token columns); beyond that an extra n-tile would re-stream
// the Q/K/V weights and double the tensor work, so the catch-up then runs as its own
// K/V product over every layer (the materialisation's), still inside the round.
bool fuse_ctx(int T, int n_pend) { return n_pend > 0 && pad16(T + n_pend) <= 128; }

// Activation buffers of the bf16 path hold a hi/lo pair: [2][pad16(T)][K] (hi block, then
// the lo block); q and the block K/V hold [2][T][...].  The Q/K/V input xq holds
// T + n_pend rows per block when the pending rows are fused (the block rows, then the
// pending context rows c_t); otherwise c_t goes to cmat and its raw K/V to kv_raw.
void carve_round(Carve &cv, RoundWs &w, const bd_config *c, int B, int W, int n_pend, int sms) {
  const bool fuse = fuse_ctx(B * W, n_pend);
  const int T = B * W, TP = pad16(T), Tq = T + (fuse ? n_pend : 0), TQ = pad16(Tq);
  const int e = elem_bytes(c);
  const int H = c->hidden, QD = c->n_q_heads * c->head_dim, KD = c->n_kv_heads * c->head_dim;
  size_t tiles = round_max_tiles(c, T, Tq);
  if (n_pend > 0 && !fuse) tiles = std::max(tiles, mat_max_tiles(c, n_pend));
  carve_gemm(cv, w.g, 2 * std::max(std::min(TQ, 128), pad16(std::min(n_pend, 128))), tiles, sms);
  const BridgePlan bp = c->code_width > 0 && c->conv_group == 0
                            ? bridge_plan(c->dtype, T, H, c->code_width, c->msg_width, sms)
                            : BridgePlan{};
  w.br_bar = bp.ok ? cv.take<unsigned>(5 * static_cast<size_t>(c->n_layers)) : nullptr;
  if (bp.ok) {
    w.zpart = cv.take<float>(static_cast<size_t>(bp.n_kz) * c->code_width * T);
    w.sspart = cv.take<float>(static_cast<size_t>(bp.n_kz) * T);
    w.zsq = cv.take<float>(static_cast<size_t>(T) * ((c->code_width + 127) / 128));
  } else {
    w.zpart = w.sspart = w.zsq = nullptr;
  }
  w.x = cv.take<float>(static_cast<size_t>(T) * H);
  w.feat = n_pend > 0 ? cv.take<float>(static_cast<size_t>(n_pend) * H) : nullptr;
  w.cmat = n_pend > 0 && !fuse ? cv.take<char>(static_cast<size_t>(n_pend) * H * e) : nullptr;
  w.kv_raw = n_pend > 0 && !fuse
                 ? cv.take<float>(static_cast<size_t>(n_pend) * c->n_layers * 2 * KD)
                 : nullptr;
  w.xn = cv.take<char>(static_cast<size_t>(2 * TP) * H * e);
  w.xq = cv.take<char>(static_cast<size_t>(2 * TQ) * H * e);
  w.q = cv.take<char>(static_cast<size_t>(2 * T) * QD * e);
  w.kblk = cv.take<char>(static_cast<size_t>(2 * T) * KD * e);
  w.vblk = cv.take<char>(static_cast<size_t>(2 * T) * KD * e);
  w.att = cv.take<char>(static_cast<size_t>(2 * TP) * QD * e);
  w.hmid = cv.take<char>(static_cast<size_t>(2 * TP) * c->ffn * e);
  w.rope = cv.take<float2>(static_cast<size_t>(T + n_pend) * (c->head_dim / 2));
  if (c->conv_group > 0) {
    const size_t nd = static_cast<size_t>(4) * H / c->conv_group;
    w.cdelta_a = cv.take<float>(static_cast<size_t>(Tq) * nd);
    w.cdelta_m = cv.take<float>(static_cast<size_t>(T) * nd);
    w.cz = cv.take<float>(static_cast<size_t>(T) * H);
    w.cn = cv.take<float>(static_cast<size_t>(T) * H);
  } else {
    w.cdelta_a = w.cdelta_m = w.cz = w.cn = nullptr;
  }
  if (c->code_width > 0) {
    w.r = cv.take<float>(T);
    w.z = cv.take<float>(static_cast<size_t>(T) * c->code_width);
    w.c = cv.take<char>(static_cast<size_t>(2 * TP) * c->code_width * e);
    w.pre = cv.take<float>(static_cast<size_t>(T) * 3 * c->msg_width);
    w.m = cv.take<char>(static_cast<size_t>(2 * TP) * c->msg_width * e);
  } else {
    w.r = w.z = w.pre = nullptr;
    w.c = w.m = nullptr;
  }
}

struct MatWs {
  GemmWs g;
  float *feat, *kv_raw;
  void *cmat;
  float2 *rope;
};
size_t mat_max_tiles(const bd_config *c, int n) {
  const size_t ntn = static_cast<size_t>(gemm_max_n_tiles(n));
  const size_t kv_tiles = static_cast<size_t>(std::min(c->n_layers, kMaxSegs / 2)) * 2 *
                          tiles_of(c->n_kv_heads * c->head_dim, 128);
  return std::max(tiles_of(c->hidden, 128), kv_tiles) * ntn;
}
void carve_mat(Carve &cv, MatWs &w, const bd_config *c, int n, int sms) {
  carve_gemm(cv, w.g, gemm_block_n(n), mat_max_tiles(c, n), sms);
  w.feat = cv.take<float>(static_cast<size_t>(n) * c->hidden);
  w.kv_raw = cv.take<float>(static_cast<size_t>(n) * c->n_layers * 2 * c->n_kv_heads * c->head_dim);
  w.cmat = cv.take<char>(static_cast<size_t>(n) * c->hidden * elem_bytes(c));
  w.rope = cv.take<float2>(static_cast<size_t>(n) * (c->head_dim / 2));
}

struct HeadWs {
  GemmWs g;
  float *amax_val;
  int32_t *amax_idx;
  float *topk_val;    // [m_tiles][rows][kTopK] per-tile candidate lists
  int32_t *topk_idx;
  float *topk_part_val;  // [rows][slices][kTopK] per-slice lists
  int32_t *topk_part_idx;
  void *hl;  // bf16 hi/lo pair of the hidden rows [2][pad16(rows)][H]
  unsigned *row_done;  // FP8 retrieval: [rows] rescoring counters, right after g.counters
  void *q8;          // e4m3 codes of the hidden rows [rows][H]
  int32_t *ties;     // [rows][m_tiles * kTopK] candidates tied at the selection threshold
  int32_t *cand;     // [rows][kMaxCand] selected candidates
  float *cscore;     // [rows][kMaxCand] their exact scores
};
constexpr int kMaxCand = 256;  // FP8 retrieval candidates per row
void carve_head(Carve &cv, HeadWs &w, const bd_config *c, int rows, int sms) {
  const size_t m_tiles = tiles_of(c->vocab, 128);
  const int bn = 2 * pad16(rows);
  carve_gemm(cv, w.g, bn, m_tiles, sms);
  w.row_done = cv.take<unsigned>(rows);
  w.hl = cv.take<char>(static_cast<size_t>(2 * pad16(rows)) * c->hidden * 2);
  w.amax_val = cv.take<float>(m_tiles * rows);
  w.amax_idx = cv.take<int32_t>(m_tiles * rows);
  w.topk_val = cv.take<float>(m_tiles * rows * kTopK);
  w.topk_idx = cv.take<int32_t>(m_tiles * rows * kTopK);
  const size_t slices = static_cast<size_t>(topk_slices(static_cast<int>(m_tiles)));
  w.topk_part_val = cv.take<float>(rows * slices * kTopK);
  w.topk_part_idx = cv.take<int32_t>(rows * slices * kTopK);
  w.q8 = cv.take<char>(static_cast<size_t>(rows) * c->hidden);
  w.ties = cv.take<int32_t>(rows * m_tiles * kTopK);
  w.cand = cv.take<int32_t>(static_cast<size_t>(rows) * kMaxCand);
  w.cscore = cv.take<float>(static_cast<size_t>(rows) * kMaxCand);
}

// Last-write refinement of B requests, K mask rows, kc candidates per row:
// n = B (K - 1) kc predecessor pairs.
struct TailWs {
  GemmWs g;
  void *cg;       // [n][Rc] predecessor candidates' codebook rows
  float *pre2;    // [n][2 Mc] (G_p C_s, A C_s)
  void *m;        // [2][pad16(n)][Mc] refined message, hi+lo pair
  float *delta;   // [n][H] W_L m
  float *table;   // [B][K-1][kc][kc] when the caller wants no copy
};
int tail_pairs(int B, int K, int kc) { return B * (K - 1) * kc; }
void carve_tail(Carve &cv, TailWs &w, const bd_config *c, int B, int K, int kc, int sms) {
  const int n = tail_pairs(B, K, kc);
  const int e = elem_bytes(c);
  const int np = pad16(n > 0 ? n : 1);
  // GEMM tiles: the gate/value maps (2 Mc rows) over n columns, the write (H rows) over
  // n columns in 128-column tiles
  const size_t ntn = static_cast<size_t>((np + 127) / 128);
  const size_t tiles = std::max(2 * tiles_of(c->msg_width, 128) * ((n + 255) / 256 + 1),
                                tiles_of(c->hidden, 128) * ntn);
  carve_gemm(cv, w.g, 256, tiles, sms);
  w.cg = cv.take<char>(static_cast<size_t>(np) * c->code_width * e);
  w.pre2 = cv.take<float>(static_cast<size_t>(np) * 2 * c->msg_width);
  w.m = cv.take<char>(static_cast<size_t>(2 * np) * c->msg_width * e);
  w.delta = cv.take<float>(static_cast<size_t>(np) * c->hidden);
  w.table = cv.take<float>(static_cast<size_t>(B) * (K - 1) * kc * kc);
}

GemmScratch scratch_of(const GemmWs &g) {
  return GemmScratch{g.partials, g.partial_floats, g.counters, g.n_counters};
}

// The call's tile counters (arrival and done), zeroed by its first kernel.
ZeroSpan counters_of(const GemmWs &g) { return ZeroSpan{g.counters, 2 * g.n_counters}; }

GemmPlan make_plan(const bd_config *c, const void *x, int n_tok, int K) {
  GemmPlan p;
  memset(&p, 0, sizeof p);
  p.dtype = c->dtype == BD_BF16 ? 0 : 1;
  p.x = x;
  p.n_tokens = n_tok;
  p.K = K;
  p.args.vocab = c->vocab;
  return p;
}
void add_w(GemmPlan &p, const void *ptr, int rows, const uint8_t *packed_base = nullptr,
           size_t packed_off = 0) {
  p.w[p.n_w].ptr = ptr;
  p.w[p.n_w].rows = rows;
  p.w[p.n_w].packed = packed_base ? packed_base + packed_off : nullptr;
  ++p.n_w;
}

}  // namespace

namespace bd {
// The configuration checks every entry point applies, for entry points in other files.
std::string validate_config(const bd_config *c) { return check_config(c); }
}  // namespace bd

// S2 for n context rows c (config dtype, [n][H]): every layer's raw K|V in one product
// (up to kMaxSegs/2 layers per launch) into kv_raw [n][L*2*Hkv*D], then head norm + RoPE +
// ring scatter of every layer in one launch (row r at position pos[r] of ring row
// req[r] < n_req, stored only inside the final live window of frontier[req[r]]).
static bd_status enqueue_ctx_kv(const bd_config *cfg, const bd_weights *w, const bd_kv_cache *kv,
                                const void *cmat, int n_rows, float *kv_raw, const float2 *rope,
                                const int32_t *row_request, const int64_t *row_pos,
                                const int64_t *ctx_frontier, int n_req, int min_back,
                                const GemmScratch &sc, cudaStream_t s) {
  const int H = cfg->hidden, D = cfg->head_dim, KD = cfg->n_kv_heads * D;
  const uint8_t *pk = static_cast<const uint8_t *>(w->packed);
  const PackedLayout PL = packed_layout(cfg);
  const int ldkv = cfg->n_layers * 2 * KD;
  for (int l0 = 0; l0 < cfg->n_layers; l0 += kMaxSegs / 2) {
    const int l1 = std::min(cfg->n_layers, l0 + kMaxSegs / 2);
    GemmPlan p = make_plan(cfg, cmat, n_rows, H);
    if (pk && packed_f16(cfg)) p.dtype = GT_F16;  // the packed W_k|W_v are fp16, c_t too
    p.args.epi = EPI_STORE_F32;
    p.args.out_f32 = kv_raw;
    p.args.ld_out = ldkv;
    for (int l = l0; l < l1; ++l) {
      const int sk = p.n_w;
      add_w(p, w->layer[l].wk, KD, pk, PL.wk[l]);
      add_w(p, w->layer[l].wv, KD, pk, PL.wv[l]);
      p.args.seg[sk].out_col = l * 2 * KD;
      p.args.seg[sk + 1].out_col = l * 2 * KD + KD;
    }
    BD_TRY(launch_gemm(p, sc, s));
  }
  HeadPostArgs h;
  memset(&h, 0, sizeof h);
  h.raw = kv_raw;
  h.ld_raw = ldkv;
  h.D = D;
  h.n_kv_heads = cfg->n_kv_heads;
  h.n_req = n_req;
  h.eps = cfg->eps;
  h.rope = rope;
  h.row_req = row_request;
  h.row_pos = row_pos;
  h.frontier = ctx_frontier;
  h.min_back = min_back;
  int n_segs = 0;
  for (int l = 0; l < cfg->n_layers; ++l) {
    HeadSeg &k = h.seg[n_segs++];
    k.kind = HK_K;
    k.col0 = l * 2 * KD;
    k.n_heads = cfg->n_kv_heads;
    k.cap = cfg->ring_capacity[l];
    k.norm = w->layer[l].k_norm;
    k.dst = kv->k[l];
    HeadSeg &v = h.seg[n_segs++];
    v = k;
    v.kind = HK_V;
    v.col0 = l * 2 * KD + KD;
    v.norm = nullptr;
    v.dst = kv->v[l];
  }
  h.rows = n_rows;
  h.n_segs = n_segs;
  h.total_heads = 2 * cfg->n_layers * cfg->n_kv_heads;
  BD_TRY(launch_head_post(cfg->dtype, h, s));
  return BD_OK;
}

// ====================================================================== C ABI
extern "C" {

int bd_abi_version(void) { return BD_ABI_VERSION; }

const char *bd_last_error(void) { return t_last_error.c_str(); }

uint64_t bd_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

size_t bd_workspace_bytes(const bd_config *cfg, int b_max, int max_masks, int max_ctx_rows) {
  if (!check_config(cfg).empty()) return 0;
  if (b_max < 1 || b_max > kMaxB || max_masks < 1 || max_masks > kMaxMasks || max_ctx_rows < 1)
    return 0;
  const int sms = sms_for_sizing();
  size_t need = 0;
  for (int B = 1; B <= b_max; ++B) {
    Carve cv;
    RoundWs w;
    carve_round(cv, w, cfg, B, max_masks + 1, kMaxPendPerReq * B, sms);
    need = std::max(need, cv.off);
    Carve ch;
    HeadWs hw;
    carve_head(ch, hw, cfg, B * max_masks, sms);
    need = std::max(need, ch.off);
    if (cfg->code_width > 0 && max_masks >= 2) {
      Carve ct;
      TailWs tw;
      carve_tail(ct, tw, cfg, B, max_masks, BD_TOPK_MAX, sms);
      need = std::max(need, ct.off);
    }
  }
  Carve cm;
  MatWs mw;
  carve_mat(cm, mw, cfg, max_ctx_rows, sms);
  need = std::max(need, cm.off);
  return need;
}

size_t bd_packed_bytes(const bd_config *cfg) {
  if (!check_config(cfg).empty()) return 0;
  return packed_layout(cfg).total;
}

bd_status bd_pack_weights(const bd_config *cfg, const bd_weights *w, void *packed,
                          size_t packed_bytes, void *stream_) {
  std::string e = check_config(cfg);
  if (!e.empty()) return fail(BD_ERR_INVALID_ARG, e);
  if ((e = check_weights(cfg, w)).empty() == false) return fail(BD_ERR_INVALID_ARG, e);
  if (!packed || (reinterpret_cast<uintptr_t>(packed) & 1023))
    return fail(BD_ERR_INVALID_ARG, "packed image NULL or not 1024-byte aligned");
  if (packed_bytes < packed_layout(cfg).total)
    return fail(BD_ERR_INVALID_ARG, "packed image smaller than bd_packed_bytes()");
  BD_TRY(pack_all(cfg, w, static_cast<uint8_t *>(packed), static_cast<cudaStream_t>(stream_)));
  return BD_OK;
}

bd_status bd_ctx_kv_materialize(const bd_config *cfg, const bd_weights *w, const bd_kv_cache *kv,
                                const void *target_feats, const int32_t *row_request,
                                const int64_t *row_pos, const int64_t *ctx_frontier, int n_rows,
                                void *workspace, size_t workspace_bytes, void *stream_) {
  std::string e = check_config(cfg);
  if (!e.empty()) return fail(BD_ERR_INVALID_ARG, e);
  if ((e = check_weights(cfg, w)).empty() == false) return fail(BD_ERR_INVALID_ARG, e);
  if ((e = check_kv(cfg, kv, 1)).empty() == false) return fail(BD_ERR_INVALID_ARG, e);
  if (n_rows < 1) return fail(BD_ERR_INVALID_ARG, "n_rows must be >= 1");
  if (!target_feats || !aligned16(target_feats)) return fail(BD_ERR_INVALID_ARG, "target_feats NULL or misaligned");
  if (!row_request || !row_pos || !ctx_frontier) return fail(BD_ERR_INVALID_ARG, "row_request/row_pos/ctx_frontier NULL");
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)))
    return fail(BD_ERR_WORKSPACE, "workspace NULL or not 256-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream_);
  const int sms = num_sms();
  Carve cv;
  cv.base = static_cast<char *>(workspace);
  MatWs mw;
  carve_mat(cv, mw, cfg, n_rows, sms);
  if (cv.off > workspace_bytes) return fail(BD_ERR_WORKSPACE, "workspace too small for materialisation");
  const int H = cfg->hidden, D = cfg->head_dim;
  const RopeFreq freq = rope_freq(cfg);
  const GemmScratch sc = scratch_of(mw.g);
  const uint8_t *pk = static_cast<const uint8_t *>(w->packed);
  const PackedLayout PL = packed_layout(cfg);

  BD_TRY(launch_rope_table(row_pos, n_rows, mw.rope, D / 2, freq, counters_of(mw.g), s));
  {  // S1: W_feature s_t (fp32 out), then plain_rmsnorm with context_norm
    GemmPlan p = make_plan(cfg, target_feats, n_rows, cfg->n_target_layers * H);
    add_w(p, w->w_feature, H, pk, PL.w_feature);
    p.args.epi = EPI_STORE_F32;
    p.args.out_f32 = mw.feat;
    p.args.ld_out = H;
    BD_TRY(launch_gemm(p, sc, s));
    BD_TRY(launch_rownorm(cfg->dtype, mw.feat, n_rows, H, w->context_norm, cfg->eps, NORM_PLAIN,
                          mw.cmat, nullptr, nullptr, nullptr, 1, 0, s, ConvFinish{nullptr, nullptr, nullptr, 0},
                          pk != nullptr && packed_f16(cfg)));
  }
  // S2: every layer's raw context K and V (fp32), then head norm + RoPE + ring scatter
  return enqueue_ctx_kv(cfg, w, kv, mw.cmat, n_rows, mw.kv_raw, mw.rope, row_request, row_pos,
                        ctx_frontier, kv->b_max, 0, sc, s);
}

bd_status bd_draft_round(const bd_config *cfg, const bd_weights *w, const bd_kv_cache *kv,
                         const int32_t *anchor_ids, const int64_t *frontier, int B, int n_masks,
                         float *head_in, float *hidden_out, float *layers_out, float *tail_state,
                         const bd_pending *pending, void *workspace, size_t workspace_bytes,
                         void *stream_) {
  std::string e = check_config(cfg);
  if (!e.empty()) return fail(BD_ERR_INVALID_ARG, e);
  if (B < 1 || B > kMaxB) return fail(BD_ERR_INVALID_ARG, "B must be in 1..8");
  if (n_masks < 1 || n_masks > kMaxMasks) return fail(BD_ERR_INVALID_ARG, "n_masks must be in 1..15");
  if ((e = check_weights(cfg, w)).empty() == false) return fail(BD_ERR_INVALID_ARG, e);
  if ((e = check_kv(cfg, kv, B)).empty() == false) return fail(BD_ERR_INVALID_ARG, e);
  if (!anchor_ids || !frontier) return fail(BD_ERR_INVALID_ARG, "anchor_ids/frontier NULL");
  if (!head_in || !aligned16(head_in)) return fail(BD_ERR_INVALID_ARG, "head_in NULL or misaligned");
  if (tail_state && cfg->code_width == 0)
    return fail(BD_ERR_INVALID_ARG, "tail_state needs the injection bridge (code_width > 0)");
  const int n_pend = pending ? pending->n_rows : 0;
  if (pending) {
    if (n_pend < 0 || n_pend > kMaxPendPerReq * B)
      return fail(BD_ERR_INVALID_ARG, "pending->n_rows must be in 0..16*B");
    if (n_pend > 0 && (!pending->feats || !aligned16(pending->feats) || !pending->request || !pending->pos))
      return fail(BD_ERR_INVALID_ARG, "pending feats/request/pos NULL or misaligned");
  }
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)))
    return fail(BD_ERR_WORKSPACE, "workspace NULL or not 256-byte aligned");
  const int W = n_masks + 1, T = B * W, TP = pad16(T);
  const int G = cfg->n_q_heads / cfg->n_kv_heads;
  if (cfg->dtype == BD_BF16 && G * W > attention_rows_max())
    return fail(BD_ERR_UNSUPPORTED, "(n_q_heads/n_kv_heads)*(n_masks+1) must be <= 64");
  for (int l = 0; l < cfg->n_layers; ++l)
    if (cfg->dtype == BD_F32 && att_max_keys(cfg, l, W) > 48 * 1024)
      return fail(BD_ERR_UNSUPPORTED, "fp32 attention supports at most 49152 keys per layer");
  cudaStream_t s = static_cast<cudaStream_t>(stream_);
  t_timing.next = 0;
  const int sms = num_sms();
  Carve cv;
  cv.base = static_cast<char *>(workspace);
  RoundWs rw;
  carve_round(cv, rw, cfg, B, W, n_pend, sms);
  if (cv.off > workspace_bytes) return fail(BD_ERR_WORKSPACE, "workspace too small for this round");
  const bool fuse = fuse_ctx(T, n_pend);
  const int Tq = T + (fuse ? n_pend : 0), TQ = pad16(Tq);

  const int H = cfg->hidden, D = cfg->head_dim;
  const int QD = cfg->n_q_heads * D, KD = cfg->n_kv_heads * D;
  const RopeFreq freq = rope_freq(cfg);
  const GemmScratch sc = scratch_of(rw.g);
  const int dt = cfg->dtype;
  const bool split = dt == BD_BF16;
  const uint8_t *pk = static_cast<const uint8_t *>(w->packed);
  const PackedLayout PL = packed_layout(cfg);  // bf16 activations enter the GEMMs as hi+lo pairs
  auto lo = [&](int K) -> size_t { return split ? static_cast<size_t>(TP) * K : 0; };

  // S3: block input rows and the RoPE table of positions F_b + i
  // the first kernel clears the GEMM tile counters (and the fused bridge's barrier
  // counters, carved right after them)
  const ZeroSpan zero{rw.g.counters, rw.br_bar ? static_cast<size_t>(rw.br_bar - rw.g.counters) +
                                                     5 * cfg->n_layers
                                               : 2 * rw.g.n_counters};
  BD_TRY(launch_round_prep(dt, w->embed_head, H, cfg->vocab, anchor_ids, frontier, B, W,
                           cfg->mask_token_id, rw.x, rw.rope, D / 2, freq,
                           n_pend > 0 ? pending->pos : nullptr, n_pend, zero, s));
  // packed image of a bf16 config: the Q/K/V, W_o, MLP and head products (and the context
  // rows' K/V products) take fp16 operands: one 16-bit operand instead of a bf16 hi+lo pair
  const bool f16 = pk != nullptr && packed_f16(cfg);
  const ConvFinish no_fin{nullptr, nullptr, nullptr, 0};
  const size_t lo_q = split && !f16 ? static_cast<size_t>(TQ) * H : 0;  // lo block of xq
  if (n_pend > 0) {  // S1 of the catch-up: c_t = plain_rmsnorm(W_feature s_t)
    GemmPlan p = make_plan(cfg, pending->feats, n_pend, cfg->n_target_layers * H);
    add_w(p, w->w_feature, H, pk, PL.w_feature);
    p.args.epi = EPI_STORE_F32;
    p.args.out_f32 = rw.feat;
    p.args.ld_out = H;
    BD_TRY(launch_gemm(p, sc, s));
    if (fuse) {  // into rows T.. of xq, with a zero lo part
      char *ctx_rows = static_cast<char *>(rw.xq) + static_cast<size_t>(T) * H * elem_bytes(cfg);
      BD_TRY(launch_rownorm(dt, rw.feat, n_pend, H, w->context_norm, cfg->eps, NORM_CTX, ctx_rows,
                            nullptr, nullptr, nullptr, 1, lo_q, s, no_fin, f16));
    } else {  // S2 of the catch-up as its own product over every layer
      BD_TRY(launch_rownorm(dt, rw.feat, n_pend, H, w->context_norm, cfg->eps, NORM_PLAIN, rw.cmat,
                            nullptr, nullptr, nullptr, 1, 0, s, no_fin, f16));
      const bd_status st = enqueue_ctx_kv(cfg, w, kv, rw.cmat, n_pend, rw.kv_raw,
                                          rw.rope + static_cast<size_t>(T) * (D / 2),
                                          pending->request, pending->pos, frontier, B,
                                          kMaxPendPerReq, sc, s);
      if (st != BD_OK) return st;
    }
  }
  // DFlash2 convolution: each branch's delta = W_delta X comes from its normalised input;
  // Conv_0 prepares that input for the branch's products, and Conv_1 of the branch output
  // is added to the residual by the next row norm (ConvFinish), which writes x back.
  const bool conv = cfg->conv_group > 0;
  const int gw = cfg->conv_group, ND = conv ? 4 * H / gw : 0;
  const bool mlp16 = f16;
  ConvFinish fin = no_fin;  // the previous layer's MLP finish, not yet added to x
  int copy_layer = -1;      // layer whose layers_out copy waits for that finish
  auto delta_gemm = [&](const void *xin, int rows, const void *wd, size_t packed_off,
                        float *out) -> std::string {
    GemmPlan p = make_plan(cfg, xin, rows, H);
    p.split = split && !f16;
    if (f16) p.dtype = GT_F16;
    add_w(p, wd, ND, pk, packed_off);
    p.args.epi = EPI_STORE_F32;
    p.args.out_f32 = out;
    p.args.ld_out = ND;
    return launch_gemm(p, sc, s);
  };
  auto copy_layer_out = [&](int l) -> std::string {
    return launch_copy_f32(rw.x, layers_out + static_cast<size_t>(l) * T * H,
                           static_cast<size_t>(T) * H, s);
  };
  for (int l = 0; l < cfg->n_layers; ++l) {
    const bd_layer_weights &L = w->layer[l];
    // S4: n = rmsnorm(x); q, k, v with head norm + RoPE.  The pending context rows ride
    // along in the same product: their K/V (S2) use the same W_k, W_v tiles.
    BD_TRY(launch_rownorm(dt, rw.x, T, H, L.in_norm, cfg->eps, NORM_PLAIN, rw.xq, nullptr,
                          conv ? rw.cn : nullptr, nullptr, W, lo_q, s, fin, f16));
    fin = no_fin;
    if (copy_layer >= 0) {
      BD_TRY(copy_layer_out(copy_layer));
      copy_layer = -1;
    }
    if (conv) {  // delta_a (over every xq row, so the split layout matches), then Conv_0(n)
      BD_TRY(delta_gemm(rw.xq, Tq, L.conv_delta_a, PL.conv_a[l], rw.cdelta_a));
      BD_TRY(launch_conv_prepare(dt, rw.cn, rw.cdelta_a, L.conv_base_a, T, H, gw, W, rw.xq, lo_q, s, f16));
    }
    {
      GemmPlan p = make_plan(cfg, rw.xq, Tq, H);
      p.split = split && !f16;
      if (f16) p.dtype = GT_F16;
      add_w(p, L.wq, QD, pk, PL.wq[l]);
      add_w(p, L.wk, KD, pk, PL.wk[l]);
      add_w(p, L.wv, KD, pk, PL.wv[l]);
      // S4's head post-processing (head RMSNorm + RoPE, queries scaled by log2(e)/sqrt(D)
      // so that the attention's scores come out in log2 units) in the product's epilogue:
      // the attention takes the queries and the block's keys/values as bf16 hi+lo planes,
      // and the pending rows' keys/values go to the rings before the attention reads them
      QkvPost &e = p.args.qkv;
      e.D = D;
      e.W = W;
      e.n_q_heads = cfg->n_q_heads;
      e.n_kv_heads = cfg->n_kv_heads;
      e.T = T;
      e.n_pend = fuse ? n_pend : 0;
      e.out_f32 = dt == BD_BF16 ? 0 : 1;
      e.eps = cfg->eps;
      e.q_scale = split ? static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D))) : 0.f;
      e.rope = rw.rope;
      e.q_norm = L.q_norm;
      e.k_norm = L.k_norm;
      e.q = rw.q;
      e.kblk = rw.kblk;
      e.vblk = rw.vblk;
      e.q_lo = split ? static_cast<size_t>(T) * QD : 0;
      e.kv_lo = split ? static_cast<size_t>(T) * KD : 0;
      if (fuse) {
        e.n_req = B;
        e.min_back = kMaxPendPerReq;
        e.cap = cfg->ring_capacity[l];
        e.kring = kv->k[l];
        e.vring = kv->v[l];
        e.row_req = pending->request;
        e.row_pos = pending->pos;
        e.frontier = frontier;
      }
      p.args.epi = EPI_QKV;
      BD_TIMED(BD_TIME_QKV, launch_gemm(p, sc, s));
    }
    // S5: block attention over the ring context and the block
    {
      AttArgs a;
      memset(&a, 0, sizeof a);
      a.q = rw.q;
      a.ring_k = kv->k[l];
      a.ring_v = kv->v[l];
      a.blk_k = rw.kblk;
      a.blk_v = rw.vblk;
      a.out = rw.att;
      a.frontier = frontier;
      a.B = B;
      a.W = W;
      a.n_q_heads = cfg->n_q_heads;
      a.n_kv_heads = cfg->n_kv_heads;
      a.head_dim = D;
      a.window = cfg->window[l];
      a.cap = cfg->ring_capacity[l];
      a.causal = cfg->block_mask == BD_BLOCK_CAUSAL ? 1 : 0;
      a.n_splits = dt == BD_BF16 ? att_splits(cfg, l, B, W, sms) : 1;
      a.n_guard = n_pend > 0 ? kMaxPendPerReq : 0;
      a.max_keys = att_max_keys(cfg, l, W);
      a.q_lo = split ? static_cast<size_t>(T) * QD : 0;
      a.blk_lo = split ? static_cast<size_t>(T) * KD : 0;
      a.out_lo = f16 ? 0 : lo(QD);
      a.out_f16 = f16 ? 1 : 0;  // W_o takes fp16 operands with the packed image
      BD_TIMED(BD_TIME_ATTENTION, launch_attention(a, dt, s));
    }
    // S6: y = x + W_o a (in place; with the convolution W_o a goes to cz and the next
    // row norm adds Conv_1 of it)
    {
      GemmPlan p = make_plan(cfg, rw.att, T, QD);
      p.split = split && !f16;
      if (f16) p.dtype = GT_F16;
      add_w(p, L.wo, H, pk, PL.wo[l]);
      p.args.epi = conv ? EPI_STORE_F32 : EPI_RESID_F32;
      p.args.out_f32 = conv ? rw.cz : rw.x;
      p.args.ld_out = H;
      BD_TIMED(BD_TIME_WO, launch_gemm(p, sc, s));
    }
    // S7: m = rmsnorm(y); x = y + W_down(SiLU(W_gate m) * W_up m).  With the packed image
    // (fp16 MLP matrices) m and the SwiGLU product are fp16 operands, else bf16 pairs.
    BD_TRY(launch_rownorm(dt, rw.x, T, H, L.post_norm, cfg->eps, NORM_PLAIN, rw.xn, nullptr,
                          conv ? rw.cn : nullptr, nullptr, W, mlp16 ? 0 : lo(H), s,
                          conv ? ConvFinish{rw.cz, rw.cdelta_a, L.conv_base_a, gw} : no_fin, mlp16));
    if (conv) {  // delta_m, then Conv_0(m)
      if (mlp16) {
        GemmPlan p = make_plan(cfg, rw.xn, T, H);
        p.dtype = GT_F16;
        add_w(p, L.conv_delta_m, ND, pk, PL.conv_m[l]);
        p.args.epi = EPI_STORE_F32;
        p.args.out_f32 = rw.cdelta_m;
        p.args.ld_out = ND;
        BD_TRY(launch_gemm(p, sc, s));
      } else {
        BD_TRY(delta_gemm(rw.xn, T, L.conv_delta_m, PL.conv_m[l], rw.cdelta_m));
      }
      BD_TRY(launch_conv_prepare(dt, rw.cn, rw.cdelta_m, L.conv_base_m, T, H, gw, W, rw.xn,
                                 mlp16 ? 0 : lo(H), s, mlp16));
    }
    {
      GemmPlan p = make_plan(cfg, rw.xn, T, H);
      p.split = split && !mlp16;
      if (mlp16) p.dtype = GT_F16;
      add_w(p, L.w_gate, cfg->ffn, pk, PL.gate_up[l]);
      add_w(p, L.w_up, cfg->ffn, pk, PL.gate_up[l]);
      p.pair_mode = true;
      p.args.epi = EPI_SWIGLU;
      p.args.out_act = rw.hmid;
      p.args.ld_act = cfg->ffn;
      p.args.act_lo = mlp16 ? 0 : static_cast<long long>(lo(cfg->ffn));
      BD_TIMED(BD_TIME_GATE_UP, launch_gemm(p, sc, s));
    }
    {
      GemmPlan p = make_plan(cfg, rw.hmid, T, cfg->ffn);
      p.split = split && !mlp16;
      if (mlp16) p.dtype = GT_F16;
      add_w(p, L.w_down, H, pk, PL.w_down[l]);
      p.args.epi = conv ? EPI_STORE_F32 : EPI_RESID_F32;
      p.args.out_f32 = conv ? rw.cz : rw.x;
      p.args.ld_out = H;
      BD_TIMED(BD_TIME_DOWN, launch_gemm(p, sc, s));
    }
    if (conv) fin = ConvFinish{rw.cz, rw.cdelta_m, L.conv_base_m, gw};
    if (cfg->code_width > 0 && rw.br_bar && pk) {  // S8 + S9 in one launch (small blocks)
      const BridgePlan bp = bridge_plan(dt, T, H, cfg->code_width, cfg->msg_width, sms);
      BridgeArgs ba;
      memset(&ba, 0, sizeof ba);
      ba.x = rw.x;
      ba.pk_r = pk + PL.r_read[l];
      ba.pk_w = pk + PL.w_write[l];
      ba.pk_g = pk + PL.g_recv;
      ba.pk_gp = pk + PL.g_pred;
      ba.pk_a = pk + PL.a_val;
      ba.gate_bias = static_cast<const __nv_bfloat16 *>(w->gate_bias);
      ba.codebook = static_cast<const __nv_bfloat16 *>(w->codebook);
      ba.anchors = anchor_ids;
      ba.r = rw.r;
      ba.zpart = rw.zpart;
      ba.sspart = rw.sspart;
      ba.zc = static_cast<__half *>(rw.c);
      ba.zsq = rw.zsq;
      ba.m = static_cast<__half *>(rw.m);
      ba.tail = tail_state && l == cfg->n_layers - 1 ? tail_state : nullptr;
      ba.bar = rw.br_bar + 5 * l;
      ba.T = T;
      ba.W = W;
      ba.H = H;
      ba.Rc = cfg->code_width;
      ba.Mc = cfg->msg_width;
      ba.V = cfg->vocab;
      ba.n_kz = bp.n_kz;
      ba.kz = bp.kz;
      ba.n1 = bp.n1;
      ba.n3 = bp.n3;
      ba.p3_boxes = bp.p3_boxes;
      ba.off_x = bp.off_x;
      ba.off_c = bp.off_c;
      ba.off_w4 = bp.off_w4;
      ba.off_red = bp.off_red;
      ba.eps = cfg->eps;
      BD_TIMED(BD_TIME_BRIDGE, launch_bridge(ba, bp, sms, s));
    } else if (cfg->code_width > 0) {
      const int Rc = cfg->code_width, Mc = cfg->msg_width;
      // S8: r = RMS(x); z = R_l (x / (r + eps)); c = sqrt(Rc) z / (|z| + eps); anchor code
      // (with the packed image the bridge's products take single fp16 operands)
      BD_TRY(launch_rownorm(dt, rw.x, T, H, nullptr, cfg->eps, NORM_BRIDGE, rw.xn, rw.r, nullptr,
                            nullptr, W, f16 ? 0 : lo(H), s, fin, f16));
      fin = no_fin;
      {
        GemmPlan p = make_plan(cfg, rw.xn, T, H);
        p.split = split && !f16;
        if (f16) p.dtype = GT_F16;
        add_w(p, L.r_read, Rc, pk, PL.r_read[l]);
        p.args.epi = EPI_STORE_F32;
        p.args.out_f32 = rw.z;
        p.args.ld_out = Rc;
        BD_TRY(launch_gemm(p, sc, s));
      }
      BD_TRY(launch_code(dt, rw.z, T, Rc, w->codebook, anchor_ids, cfg->vocab, W, cfg->eps, rw.c,
                         f16 ? 0 : lo(Rc), s, f16));
      // S9: [G c; G_p c; A c] in one launch, gate/message, then the RMS-scaled write
      {
        GemmPlan p = make_plan(cfg, rw.c, T, Rc);
        p.split = split && !f16;
        if (f16) p.dtype = GT_F16;
        add_w(p, w->g_recv, Mc, pk, PL.g_recv);
        add_w(p, w->g_pred, Mc, pk, PL.g_pred);
        add_w(p, w->a_val, Mc, pk, PL.a_val);
        p.args.epi = EPI_STORE_F32;
        p.args.out_f32 = rw.pre;
        p.args.ld_out = 3 * Mc;
        p.args.seg[0].out_col = 0;
        p.args.seg[1].out_col = Mc;
        p.args.seg[2].out_col = 2 * Mc;
        BD_TRY(launch_gemm(p, sc, s));
      }
      BD_TRY(launch_message(dt, rw.pre, T, Mc, w->gate_bias, W, rw.m, f16 ? 0 : lo(Mc), s, f16));
      if (tail_state && l == cfg->n_layers - 1)  // the state the last-write refinement redoes
        BD_TRY(launch_tail_export(rw.x, rw.r, rw.pre, T, H, Mc, tail_state, s));
      {
        GemmPlan p = make_plan(cfg, rw.m, T, Mc);
        p.split = split && !f16;
        if (f16) p.dtype = GT_F16;
        add_w(p, L.w_write, H, pk, PL.w_write[l]);
        p.args.epi = EPI_INJECT;
        p.args.out_f32 = rw.x;
        p.args.ld_out = H;
        p.args.row_scale = rw.r;
        p.args.block_w = W;
        BD_TRY(launch_gemm(p, sc, s));
      }
    }
    if (layers_out) {
      if (fin.z)
        copy_layer = l;  // after the next row norm has added the MLP finish
      else
        BD_TRY(copy_layer_out(l));
    }
  }
  BD_TRY(launch_rownorm(dt, rw.x, T, H, w->final_norm, cfg->eps, NORM_FINAL, nullptr, nullptr,
                        hidden_out, head_in, W, 0, s, fin));
  if (copy_layer >= 0) BD_TRY(copy_layer_out(copy_layer));
  return BD_OK;
}

// Checks shared by the head entry points, carves the head workspace and enqueues the
// hi/lo split of the hidden rows (or the counter clear); returns the GEMM plan.
static bd_status head_prepare(const bd_config *cfg, const bd_weights *w, const float *hidden,
                              int rows, const int32_t *token_out, void *workspace,
                              size_t workspace_bytes, cudaStream_t s, HeadWs &hw, GemmPlan &p) {
  std::string e = check_config(cfg);
  if (!e.empty()) return fail(BD_ERR_INVALID_ARG, e);
  if (!w || !w->embed_head || !aligned16(w->embed_head))
    return fail(BD_ERR_INVALID_ARG, "embed_head NULL or misaligned");
  if (rows < 1 || rows > kMaxB * kMaxMasks) return fail(BD_ERR_INVALID_ARG, "rows must be in 1..120");
  if (!hidden || !aligned16(hidden)) return fail(BD_ERR_INVALID_ARG, "hidden NULL or misaligned");
  if (!token_out) return fail(BD_ERR_INVALID_ARG, "token_out NULL");
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)))
    return fail(BD_ERR_WORKSPACE, "workspace NULL or not 256-byte aligned");
  Carve cv;
  cv.base = static_cast<char *>(workspace);
  carve_head(cv, hw, cfg, rows, num_sms());
  if (cv.off > workspace_bytes) return fail(BD_ERR_WORKSPACE, "workspace too small for the head");
  // With the packed image the head is fp16 and the hidden rows become fp16 operands;
  // otherwise (bf16 head) a bf16 hi/lo pair of the fp32 rows, ~16 mantissa bits.
  const bool head16 = w->packed != nullptr && packed_f16(cfg);
  const bool split = cfg->dtype == BD_BF16 && !head16;
  if (head16)
    BD_TRY(launch_rows_f16(hidden, static_cast<size_t>(rows) * cfg->hidden, hw.hl, counters_of(hw.g), s));
  else if (split)
    BD_TRY(launch_split_rows(hidden, static_cast<size_t>(rows) * cfg->hidden, hw.hl,
                             static_cast<size_t>(pad16(rows)) * cfg->hidden, counters_of(hw.g), s));
  else
    BD_TRY(launch_zero(counters_of(hw.g), s));
  p = make_plan(cfg, (split || head16) ? static_cast<const void *>(hw.hl) : hidden, rows, cfg->hidden);
  p.split = split;
  if (head16) p.dtype = GT_F16;
  add_w(p, w->embed_head, cfg->vocab, static_cast<const uint8_t *>(w->packed),
        w->packed ? packed_layout(cfg).head : 0);
  return BD_OK;
}

bd_status bd_lm_head_argmax(const bd_config *cfg, const bd_weights *w, const float *hidden, int rows,
                            int32_t *token_out, float *max_logit_out, void *workspace,
                            size_t workspace_bytes, void *stream_) {
  cudaStream_t s = static_cast<cudaStream_t>(stream_);
  HeadWs hw;
  GemmPlan p;
  const bd_status st = head_prepare(cfg, w, hidden, rows, token_out, workspace, workspace_bytes, s,
                                    hw, p);
  if (st != BD_OK) return st;
  p.args.epi = EPI_ARGMAX;
  p.args.amax_val = hw.amax_val;
  p.args.amax_idx = hw.amax_idx;
  t_timing.next = 0;
  BD_TIMED(BD_TIME_HEAD, launch_gemm(p, scratch_of(hw.g), s));
  BD_TRY(launch_argmax_reduce(hw.amax_val, hw.amax_idx, static_cast<int>(tiles_of(cfg->vocab, 128)),
                              rows, token_out, max_logit_out, s));
  return BD_OK;
}

bd_status bd_lm_head_topk(const bd_config *cfg, const bd_weights *w, const float *hidden, int rows,
                          int k, int32_t *token_out, float *score_out, void *workspace,
                          size_t workspace_bytes, void *stream_) {
  if (k < 1 || k > BD_TOPK_MAX) return fail(BD_ERR_INVALID_ARG, "k must be in 1..16");
  if (cfg && cfg->vocab < k) return fail(BD_ERR_INVALID_ARG, "vocab smaller than k");
  cudaStream_t s = static_cast<cudaStream_t>(stream_);
  HeadWs hw;
  GemmPlan p;
  const bd_status st = head_prepare(cfg, w, hidden, rows, token_out, workspace, workspace_bytes, s,
                                    hw, p);
  if (st != BD_OK) return st;
  p.args.epi = EPI_TOPK;
  p.args.topk_val = hw.topk_val;
  p.args.topk_idx = hw.topk_idx;
  BD_TRY(launch_gemm(p, scratch_of(hw.g), s));
  BD_TRY(launch_topk_reduce(hw.topk_val, hw.topk_idx, static_cast<int>(tiles_of(cfg->vocab, 128)),
                            rows, k, hw.topk_part_val, hw.topk_part_idx, token_out, score_out, s));
  return BD_OK;
}

size_t bd_head_fp8_bytes(const bd_config *cfg) {
  if (!check_config(cfg).empty() || cfg->dtype != BD_BF16 || cfg->hidden % 16 != 0) return 0;
  return head_fp8_image_bytes(cfg->vocab, cfg->hidden) + static_cast<size_t>(cfg->vocab) * sizeof(float);
}

bd_status bd_pack_head_fp8(const bd_config *cfg, const bd_weights *w, void *image, size_t image_bytes,
                           void *stream_) {
  std::string e = check_config(cfg);
  if (!e.empty()) return fail(BD_ERR_INVALID_ARG, e);
  if (cfg->dtype != BD_BF16) return fail(BD_ERR_UNSUPPORTED, "the FP8 head copy is built from a bf16 head");
  if (cfg->hidden % 16 != 0) return fail(BD_ERR_UNSUPPORTED, "the FP8 head needs hidden % 16 == 0");
  if (!w || !w->embed_head || !aligned16(w->embed_head))
    return fail(BD_ERR_INVALID_ARG, "embed_head NULL or misaligned");
  if (!image || (reinterpret_cast<uintptr_t>(image) & 1023))
    return fail(BD_ERR_INVALID_ARG, "FP8 head image NULL or not 1024-byte aligned");
  if (image_bytes < bd_head_fp8_bytes(cfg))
    return fail(BD_ERR_INVALID_ARG, "FP8 head image smaller than bd_head_fp8_bytes()");
  BD_TRY(launch_head_fp8_pack(w->embed_head, cfg->vocab, cfg->hidden, image,
                              static_cast<cudaStream_t>(stream_)));
  return BD_OK;
}

bd_status bd_lm_head_topk_fp8(const bd_config *cfg, const bd_weights *w, const void *head_fp8,
                              const float *hidden, int rows, int n_cand, int k, int32_t *token_out,
                              float *score_out, void *workspace, size_t workspace_bytes,
                              void *stream_) {
  std::string e = check_config(cfg);
  if (!e.empty()) return fail(BD_ERR_INVALID_ARG, e);
  if (cfg->dtype != BD_BF16) return fail(BD_ERR_UNSUPPORTED, "FP8 retrieval needs a bf16 head");
  if (cfg->hidden % 16 != 0) return fail(BD_ERR_UNSUPPORTED, "FP8 retrieval needs hidden % 16 == 0");
  const int V = cfg->vocab, H = cfg->hidden;
  const int m_tiles = static_cast<int>(tiles_of(V, 128));
  if (select_cand_smem(m_tiles) > 200 * 1024) return fail(BD_ERR_UNSUPPORTED, "vocab too large for FP8 retrieval");
  if (k < 1 || k > BD_TOPK_MAX) return fail(BD_ERR_INVALID_ARG, "k must be in 1..16");
  if (n_cand < k || n_cand > kMaxCand || n_cand > V || n_cand > m_tiles * kTopK)
    return fail(BD_ERR_INVALID_ARG, "n_cand must be in k..256 and at most vocab");
  if (rows < 1 || rows > kMaxB * kMaxMasks) return fail(BD_ERR_INVALID_ARG, "rows must be in 1..120");
  if (!w || !w->embed_head || !aligned16(w->embed_head))
    return fail(BD_ERR_INVALID_ARG, "embed_head NULL or misaligned");
  if (!head_fp8 || (reinterpret_cast<uintptr_t>(head_fp8) & 1023))
    return fail(BD_ERR_INVALID_ARG, "FP8 head image NULL or not 1024-byte aligned");
  if (!hidden || !aligned16(hidden)) return fail(BD_ERR_INVALID_ARG, "hidden NULL or misaligned");
  if (!token_out) return fail(BD_ERR_INVALID_ARG, "token_out NULL");
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)))
    return fail(BD_ERR_WORKSPACE, "workspace NULL or not 256-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream_);
  Carve cv;
  cv.base = static_cast<char *>(workspace);
  HeadWs hw;
  carve_head(cv, hw, cfg, rows, num_sms());
  if (cv.off > workspace_bytes) return fail(BD_ERR_WORKSPACE, "workspace too small for the head");
  // the hidden rows' codes (this first kernel also clears the GEMM tile counters and the
  // rescoring counters, carved right after them)
  const ZeroSpan zero{hw.g.counters, static_cast<size_t>(hw.row_done - hw.g.counters) + rows};
  BD_TRY(launch_code_rows(hidden, rows, H, hw.q8, zero, s));
  GemmPlan p = make_plan(cfg, hw.q8, rows, H);
  p.dtype = GT_E4M3;
  add_w(p, w->embed_head, V, static_cast<const uint8_t *>(head_fp8), 0);
  p.args.epi = EPI_TOPK;
  p.args.topk_val = hw.topk_val;
  p.args.topk_idx = hw.topk_idx;
  p.args.wscale = reinterpret_cast<const float *>(static_cast<const char *>(head_fp8) +
                                                  head_fp8_image_bytes(V, H));
  BD_TRY(launch_gemm(p, scratch_of(hw.g), s));
  BD_TRY(launch_select_cand(hw.topk_val, hw.topk_idx, m_tiles, rows, n_cand, hw.ties, hw.cand, s));
  BD_TRY(launch_rescore(w->embed_head, V, H, hidden, hw.cand, rows, n_cand, k, hw.cscore,
                        hw.row_done, token_out, score_out, s));
  return BD_OK;
}

bd_status bd_refine_tail(const bd_config *cfg, const bd_weights *w, const float *tail_state,
                         const int32_t *cand_ids, const float *cand_scores, int B, int n_masks, int kc,
                         int32_t *token_out, int32_t *pick_out, float *table_out, void *workspace,
                         size_t workspace_bytes, void *stream_) {
  std::string e = check_config(cfg);
  if (!e.empty()) return fail(BD_ERR_INVALID_ARG, e);
  if (cfg->code_width == 0) return fail(BD_ERR_INVALID_ARG, "the refinement needs the injection bridge");
  if (B < 1 || B > kMaxB) return fail(BD_ERR_INVALID_ARG, "B must be in 1..8");
  if (n_masks < 2 || n_masks > kMaxMasks) return fail(BD_ERR_INVALID_ARG, "n_masks must be in 2..15");
  if (kc < 1 || kc > BD_TOPK_MAX || kc > cfg->vocab) return fail(BD_ERR_INVALID_ARG, "kc must be in 1..16");
  if ((e = check_weights(cfg, w)).empty() == false) return fail(BD_ERR_INVALID_ARG, e);
  if (!tail_state || !cand_ids || !cand_scores || !token_out)
    return fail(BD_ERR_INVALID_ARG, "tail_state, cand_ids, cand_scores and token_out are required");
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)))
    return fail(BD_ERR_WORKSPACE, "workspace NULL or not 256-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream_);
  const int K = n_masks, W = K + 1, T = B * W, H = cfg->hidden;
  const int Rc = cfg->code_width, Mc = cfg->msg_width, dt = cfg->dtype;
  const int n = tail_pairs(B, K, kc);
  Carve cv;
  cv.base = static_cast<char *>(workspace);
  TailWs tw;
  carve_tail(cv, tw, cfg, B, K, kc, num_sms());
  if (cv.off > workspace_bytes) return fail(BD_ERR_WORKSPACE, "workspace too small for the refinement");
  const float *u = tail_state;
  const float *r = tail_state + static_cast<size_t>(T) * H;
  const float *gc = r + T;
  const uint8_t *pk = static_cast<const uint8_t *>(w->packed);
  const PackedLayout PL = packed_layout(cfg);
  float *table = table_out ? table_out : tw.table;

  // the packed image holds the bridge matrices as fp16: fp16 operands on both sides
  const bool f16 = pk != nullptr && packed_f16(cfg);
  BD_TRY(launch_zero(counters_of(tw.g), s));
  BD_TRY(launch_tail_gather(dt, w->codebook, cfg->vocab, Rc, cand_ids, K, kc, n, tw.cg, s, f16));
  {  // G_p C_s and A C_s for every predecessor candidate (codebook rows are exact inputs)
    GemmPlan p = make_plan(cfg, tw.cg, n, Rc);
    if (f16) p.dtype = GT_F16;
    add_w(p, w->g_pred, Mc, pk, PL.g_pred);
    add_w(p, w->a_val, Mc, pk, PL.a_val);
    p.args.epi = EPI_STORE_F32;
    p.args.out_f32 = tw.pre2;
    p.args.ld_out = 2 * Mc;
    p.args.seg[0].out_col = 0;
    p.args.seg[1].out_col = Mc;
    BD_TRY(launch_gemm(p, scratch_of(tw.g), s));
  }
  const bool split = dt == BD_BF16 && !f16;
  const size_t lo_m = split ? static_cast<size_t>(pad16(n)) * Mc : 0;
  BD_TRY(launch_tail_message(dt, tw.pre2, gc, w->gate_bias, K, W, kc, Mc,
                             std::sqrt(static_cast<float>(Rc)), n, tw.m, lo_m, s, f16));
  {  // delta = W_L m, the refined write before its RMS scale
    GemmPlan p = make_plan(cfg, tw.m, n, Mc);
    p.split = split;
    if (f16) p.dtype = GT_F16;
    add_w(p, w->layer[cfg->n_layers - 1].w_write, H, pk, PL.w_write[cfg->n_layers - 1]);
    p.args.epi = EPI_STORE_F32;
    p.args.out_f32 = tw.delta;
    p.args.ld_out = H;
    BD_TRY(launch_gemm(p, scratch_of(tw.g), s));
  }
  BD_TRY(launch_tail_scores(dt, u, r, tw.delta, w->embed_head, w->final_norm, cand_ids, B, K, W, kc, H,
                            cfg->vocab, cfg->eps, table, s));
  BD_TRY(launch_tail_walk(table, cand_scores, cand_ids, B, K, kc, token_out, pick_out, s));
  return BD_OK;
}

bd_status bd_selftest_wait(const unsigned *flag, int limit_us, void *stream_) {
  if (!flag || (reinterpret_cast<uintptr_t>(flag) & 3)) return fail(BD_ERR_INVALID_ARG, "flag NULL or misaligned");
  if (limit_us < 1 || limit_us > 2000000) return fail(BD_ERR_INVALID_ARG, "limit_us must be in 1..2000000");
  BD_TRY(launch_wait_selftest(flag, static_cast<unsigned long long>(limit_us) * 1000ull,
                              static_cast<cudaStream_t>(stream_)));
  return BD_OK;
}

bd_status bd_set_timing_events(int kind, void *const *begin, void *const *end, int n) {
  if (kind == BD_TIME_NONE) {
    t_timing = Timing();
    return BD_OK;
  }
  if (kind < BD_TIME_QKV || kind > BD_TIME_HEAD) return fail(BD_ERR_INVALID_ARG, "unknown timing kind");
  if (n < 1 || n > BD_TIMING_MAX || !begin || !end)
    return fail(BD_ERR_INVALID_ARG, "timing events: n must be in 1..BD_TIMING_MAX with both arrays given");
  for (int i = 0; i < n; ++i)
    if (!begin[i] || !end[i]) return fail(BD_ERR_INVALID_ARG, "timing events: NULL event");
  Timing t;
  t.kind = kind;
  t.n = n;
  for (int i = 0; i < n; ++i) {
    t.begin[i] = static_cast<cudaEvent_t>(begin[i]);
    t.end[i] = static_cast<cudaEvent_t>(end[i]);
  }
  t_timing = t;
  return BD_OK;
}

bd_status bd_sync_status(void *stream_) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream_));
  if (e != cudaSuccess) return fail(BD_ERR_CUDA, std::string("stream: ") + cudaGetErrorString(e));
  const unsigned word = take_error_word_gemm() | take_error_word_att() | take_error_word_small() |
                        take_error_word_pack() | take_error_word_head8() | take_error_word_bridge();
  if (word & DEVERR_TIMEOUT) return fail(BD_ERR_DEVICE_TIMEOUT, "a bounded device wait gave up");
  if (word & DEVERR_BAD_INDEX)
    return fail(BD_ERR_INVALID_ARG, "a device-side index (token id, request or position) was out of range");
  if (word & DEVERR_RANGE)
    return fail(BD_ERR_RANGE, "a weight packed as fp16 is beyond the fp16 range (|w| > 65504)");
  if (word & DEVERR_F16)
    return fail(BD_ERR_RANGE, "an activation stored as an fp16 operand was beyond the fp16 range "
                              "(|x| > 65504) or not finite");
  return BD_OK;
}

}  // extern "C"
