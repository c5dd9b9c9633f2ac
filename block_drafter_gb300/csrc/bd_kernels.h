// Launchers of the non-GEMM kernels (attention, norms, embedding, bridge helpers).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "bd_internal.h"

namespace bd {

struct AttArgs {
  const void *q;        // [B*W, Hq*D] post-RoPE queries
  const void *ring_k;   // [b_max, Hkv, cap, D] this layer's context ring
  const void *ring_v;
  const void *blk_k;    // [B, Hkv, W, D] block keys (post-RoPE)
  const void *blk_v;
  void *out;            // [B*W, Hq*D] attention output (config dtype)
  const int64_t *frontier;  // [B]
  int B, W, n_q_heads, n_kv_heads, head_dim, window, cap, causal, n_splits, max_keys;
  int n_guard;          // context positions >= F - n_guard may be written by this round's
                        // catch-up (read only after the previous kernel has finished)
  size_t q_lo, blk_lo, out_lo;  // bf16: element offsets of the lo halves of q, blk_k/v, out
                                // (q and blk lo planes directly follow their hi planes)
  int out_f16;                  // bf16 config: the output is one fp16 plane (out_lo unused)
};

int attention_rows_max();
int attention_tile_keys();    // context keys per tile of the bf16 kernel
int attention_max_splits();   // key splits (one cluster) of a head at most
std::string launch_attention(const AttArgs &a, int dtype, cudaStream_t stream);

// theta^(-2j/D) for j < D/2, computed on the host in double precision.
struct RopeFreq {
  double inv[64];
};

// Words a call's first kernel sets to zero (the GEMM tile counters of the call): doing it
// there instead of with a memset keeps the call one chain of dependent launches.
struct ZeroSpan {
  unsigned *p;
  size_t n;
};
#ifdef __CUDACC__
// Grid-stride zeroing of a ZeroSpan (after the kernel's pdl_wait: the previous kernel,
// which may still use the words, has completed).
__device__ __forceinline__ void zero_span(ZeroSpan z) {
  for (size_t t = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; t < z.n;
       t += static_cast<size_t>(gridDim.x) * blockDim.x)
    z.p[t] = 0u;
}
#endif

// Round prologue: x[b*W+i] = embed[id] (fp32), id = anchor_b for i = 0 else MASK, the
// (cos, sin) rows of positions F_b + i (rows 0 .. B*W-1), then the rows of n_pend pending
// context positions (rows B*W ..).
std::string launch_round_prep(int dtype, const void *embed, int H, int V, const int32_t *anchors,
                              const int64_t *frontier, int B, int W, int mask_id, float *x,
                              float2 *rope, int half, const RopeFreq &freq, const int64_t *pend_pos,
                              int n_pend, ZeroSpan z, cudaStream_t s);
// (cos, sin) table of arbitrary absolute positions.
std::string launch_rope_table(const int64_t *pos, int n, float2 *rope, int half,
                              const RopeFreq &freq, ZeroSpan z, cudaStream_t s);
// Only zeroes (for calls whose first kernel is a GEMM).
std::string launch_zero(ZeroSpan z, cudaStream_t s);

enum NormMode : int {
  NORM_PLAIN = 0,   // out = gain * x / sqrt(mean(x^2) + eps)
  NORM_BRIDGE = 1,  // r = sqrt(mean(x^2)); out = x / (r + eps); r_out = r
  NORM_FINAL = 2,   // plain, plus fp32 copy and the mask-row copy for the LM head
  NORM_CTX = 3      // plain; the lo part is written as zero (c_t enters products as bf16)
};
// DFlash2 branch finish folded into the next row norm: before normalising row i, the
// kernel adds Conv_1(z)[i] (side-1 grouped convolution of the branch output z with the
// branch's delta) to x and writes the updated row back.  z == null: no finish.
struct ConvFinish {
  const float *z;      // [rows][H] branch output
  const float *delta;  // [rows][2 sides][2 taps][H / gw] (side 1 used)
  const void *base;    // [2 sides][2 taps][H], config dtype (side 1 used)
  int gw;              // group width (a multiple of 4 dividing H)
};
// Row norm of x (one CTA per row).  lo_off != 0: also write the rounding residual y - hi
// at out + lo_off (split activation).  f32_out: an fp32 copy of y, or null.
// out_f16 (bf16 config): the output is fp16 (lo_off must then be 0).
std::string launch_rownorm(int dtype, float *x, int rows, int H, const void *gain,
                           float eps, int mode, void *out, float *r_out, float *f32_out,
                           float *head_out, int W, size_t lo_off, cudaStream_t s,
                           const ConvFinish &cf = ConvFinish{nullptr, nullptr, nullptr, 0},
                           bool out_f16 = false);
// DFlash2 branch input: out = Conv_0(X) (side-0 grouped convolution of the normalised
// branch input X [rows][H] fp32 with delta [rows][2][2][H/gw]), split when lo_off != 0.
std::string launch_conv_prepare(int dtype, const float *X, const float *delta, const void *base,
                                int rows, int H, int gw, int W, void *out, size_t lo_off,
                                cudaStream_t s, bool out_f16 = false);
// fp32 -> bf16 hi (dst) and lo (dst + lo_off) of n elements.
std::string launch_split_rows(const float *src, size_t n, void *dst, size_t lo_off, ZeroSpan z,
                              cudaStream_t s);
// fp32 -> fp16 of n elements.
std::string launch_rows_f16(const float *src, size_t n, void *dst, ZeroSpan z, cudaStream_t s);

// c = sqrt(Rc) z / (||z|| + eps) for non-anchor rows; sqrt(Rc) * codebook[anchor] for anchors.
std::string launch_code(int dtype, const float *z, int rows, int Rc, const void *codebook,
                        const int32_t *anchors, int V, int W, float eps, void *c_out,
                        size_t lo_off, cudaStream_t s, bool out_f16 = false);
// m_i = sigmoid(G c_i + G_p c_{i-1} + b) * (A c_{i-1}) for i >= 1, m_0 = 0.
std::string launch_message(int dtype, const float *pre, int rows, int Mc, const void *bias,
                           int W, void *m_out, size_t lo_off, cudaStream_t s, bool out_f16 = false);
// Head post-processing of the context rows' raw fp32 key/value projections [rows, ld_raw]
// (every layer's keys and values in one row): plain_head_rmsnorm + split-half RoPE of key
// heads, a copy of value heads, rounded to the config dtype and stored in the ring slot of
// the row's position (request row_req[r], position row_pos[r]) when it lies in the final
// live window [F - cap, F).  A row whose request or position is invalid sets the
// bad-index error.
enum HeadKind : int { HK_K = 1, HK_V = 2 };
constexpr int kMaxHeadSegs = 32;
struct HeadSeg {
  int kind, col0, n_heads, cap;  // column of the segment's first head in a raw row; ring size
  const void *norm;              // [D] key-norm gain (key segments)
  void *dst;                     // ring [B][Hkv][cap][D]
};
struct HeadPostArgs {
  const float *raw;
  int ld_raw, D, n_kv_heads, n_req, rows, n_segs, total_heads;
  float eps;
  const float2 *rope;        // [rows][D/2]
  const int32_t *row_req;    // [rows]
  const int64_t *row_pos;
  const int64_t *frontier;
  int min_back;              // > 0: rows must lie in [F - min_back, F) (else an error)
  HeadSeg seg[kMaxHeadSegs];
};
std::string launch_head_post(int dtype, const HeadPostArgs &a, cudaStream_t s);

// Fused DSpine bridge for blocks of T <= 32 rows (bf16 config, packed weight image): one
// launch, one CTA per SM, phases separated by grid barriers (bar: 3 counters, zero on
// entry).  See bd_bridge.cu.
struct BridgeArgs {
  float *x;                                       // [T][H] residual, updated in place
  const uint8_t *pk_r, *pk_w;                     // packed R_l [Rc][H], W_l [H][Mc]
  const uint8_t *pk_g, *pk_gp, *pk_a;             // packed G, G_p, A [Mc][Rc]
  const __nv_bfloat16 *gate_bias;                 // [Mc] or null
  const __nv_bfloat16 *codebook;                  // [V][Rc]
  const int32_t *anchors;                         // [B]
  float *r;                                       // [T] OUT RMS of the pre-injection rows
  float *zpart, *sspart;                          // [n_kz][T][Rc], [n_kz][T]
  __half *zc;                                     // z' fp16 activation boxes (16 or 32 rows x Rc)
  float *zsq;                                     // [T][ceil(Rc / 128)]
  __half *m;                                      // message fp16 boxes (16 or 32 rows x Mc)
  float *tail;                                    // tail state export, or null
  unsigned *bar;                                  // [3] grid-barrier counters
  int T, W, H, Rc, Mc, V;
  int n_kz, kz, n1, n3, p3_boxes;                 // from the plan
  size_t off_x, off_c, off_w4, off_red;           // shared-memory areas (from the plan)
  float eps;
};
// Work split and shared-memory areas of one launch; ok = false when the shape does not fit.
struct BridgePlan {
  bool ok;
  int n_kz, kz;   // K chunks of the code read (P1 CTAs: ceil(Rc / 128) * n_kz)
  int n1, n3;     // CTAs of P1 and of P3 (Mc / 16)
  int p3_boxes;   // K boxes of the codes staged at once in P3
  size_t off_x, off_c, off_w4, off_red;  // P1 activations, P3 codes, P4 W_l rows, sums
  size_t smem;                           // dynamic shared memory of the launch
};
BridgePlan bridge_plan(int dtype, int T, int H, int Rc, int Mc, int sms);
std::string launch_bridge(const BridgeArgs &args, const BridgePlan &plan, int sms, cudaStream_t s);

// One bounded wait (the inter-CTA wait of the GEMM and attention kernels) for *flag >= 1.
std::string launch_wait_selftest(const unsigned *flag, unsigned long long limit_ns, cudaStream_t s);
// Per-row argmax over per-tile (max, lowest argmax) pairs; lowest id on ties.
std::string launch_argmax_reduce(const float *val, const int32_t *idx, int m_tiles, int rows,
                                 int32_t *tok_out, float *max_out, cudaStream_t s);
// Per-row k best (k <= kTopK) over the per-tile candidate lists [m_tiles][rows][kTopK]:
// descending score, equal scores to the lower id.  Two launches: slices of at most
// kTopKTilesPerSlice tiles per row (scratch part_* [rows][topk_slices][kTopK]), then one
// warp per row over the slices.
constexpr int kTopKTilesPerSlice = 128;
int topk_slices(int m_tiles);
std::string launch_topk_reduce(const float *val, const int32_t *idx, int m_tiles, int rows, int k,
                               float *part_val, int32_t *part_idx, int32_t *tok_out,
                               float *score_out, cudaStream_t s);
// FP8 retrieval head: the row-scaled e4m3 image of a bf16 head [V, H] (tiles of 128 rows x
// 128-byte boxes, head_fp8_image_bytes(V, H) bytes, then V fp32 row scales); the e4m3 code
// of hidden rows [rows][H]; the n_cand best of the per-tile candidate lists (radix
// selection, scratch ties [rows][m_tiles * kTopK]); exact rescoring and the k best.
size_t head_fp8_image_bytes(int V, int H);
std::string launch_head_fp8_pack(const void *E, int V, int H, void *img, cudaStream_t s);
std::string launch_code_rows(const float *h, int rows, int H, void *q, ZeroSpan z, cudaStream_t s);
size_t select_cand_smem(int m_tiles);
std::string launch_select_cand(const float *val, const int32_t *idx, int m_tiles, int rows,
                               int n_cand, int32_t *ties, int32_t *cand, cudaStream_t s);
// scores [rows][n_cand] scratch; row_done [rows] counters, zero on entry and left zero.
std::string launch_rescore(const void *E, int V, int H, const float *hidden, const int32_t *cand,
                           int rows, int n_cand, int k, float *scores, unsigned *row_done,
                           int32_t *tok_out, float *score_out, cudaStream_t s);
// Last-write refinement: state export [T][H] u | [T] r | [T][Mc] G c (from pre [T][3 Mc]),
// the predecessor candidates' codebook rows, the refined message (hi+lo pair), the
// refined scores [B][K-1][kc][kc] and the greedy walk.
std::string launch_tail_export(const float *x, const float *r, const float *pre, int T, int H,
                               int Mc, float *out, cudaStream_t s);
std::string launch_tail_gather(int dtype, const void *codebook, int V, int Rc, const int32_t *cand,
                               int K, int kc, int n_pairs, void *out, cudaStream_t s, bool out_f16 = false);
std::string launch_tail_message(int dtype, const float *pre2, const float *gc, const void *bias, int K,
                                int W, int kc, int Mc, float scale, int n_pairs, void *m_out,
                                size_t lo_off, cudaStream_t s, bool out_f16 = false);
std::string launch_tail_scores(int dtype, const float *u, const float *r, const float *delta,
                               const void *embed, const void *gain, const int32_t *cand, int B, int K,
                               int W, int kc, int H, int V, float eps, float *table, cudaStream_t s);
std::string launch_tail_walk(const float *table, const float *cand_score, const int32_t *cand, int B,
                             int K, int kc, int32_t *token_out, int32_t *pick_out, cudaStream_t s);
// Copy rows [n, H] fp32 (used for the optional per-layer residual output).
std::string launch_copy_f32(const float *src, float *dst, size_t n, cudaStream_t s);

}  // namespace bd
