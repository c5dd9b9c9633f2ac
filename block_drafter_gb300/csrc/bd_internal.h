// Internal host/device declarations shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <string>
#include <utility>

#include "blockdrafter.h"

namespace bd {

// Device error word flags (set by kernels, read and cleared by bd_sync_status()).
// DEVERR_RANGE: a weight beyond the fp16 range met the packed image's fp16 conversion;
// DEVERR_F16: an activation beyond the fp16 range (or not finite) met an fp16 operand store.
enum : unsigned { DEVERR_TIMEOUT = 1u, DEVERR_BAD_INDEX = 2u, DEVERR_RANGE = 4u, DEVERR_F16 = 8u };

// ------------------------------------------------------------------ GEMM
// D[tok, out] = X[tok, :] . W[out, :]  computed swap-AB on tcgen05: weight rows fill the
// 128-wide MMA M dimension, tokens the N dimension.  One launch streams one or more
// weight matrices ("segments") that share the activation operand X.
constexpr int kMaxSegs = 12;
constexpr int kBM = 128;
// Epilogue: kEpiSlices warps per TMEM lane quarter, each taking 16 / kEpiSlices of a
// 16-column chunk, so every SM sub-partition has kEpiSlices epilogue warps whose
// instruction latencies overlap.
constexpr int kEpiSlices = 2;
constexpr int kEpiThreads = 128 * kEpiSlices;
constexpr int kGemmThreads = 64 + kEpiThreads;  // warp 0 TMA, warp 1 MMA, then the epilogue

enum EpiMode : int {
  EPI_STORE_F32 = 0,  // out[tok*ld + out_col + row] = acc
  EPI_RESID_F32 = 1,  // out[tok*ld + row] += acc (one addition per element: deterministic)
  EPI_INJECT = 2,     // x[tok*ld + row] += scale[tok] * acc for non-anchor rows
  EPI_SWIGLU = 3,     // pair tiles: out[tok*ld_act + f] = SiLU(gate_f) * up_f
  EPI_ARGMAX = 4,     // per-tile (max, lowest argmax) over 128 vocabulary rows
  EPI_TOPK = 5,       // per-tile 16 best (score, id) over 128 vocabulary rows
  EPI_QKV = 6         // Q/K/V product: head RMSNorm + RoPE, scattered to the attention inputs
};
constexpr int kTopK = 16;  // candidates per tile and per row of the top-k head

struct GemmSeg {
  int rows;               // output rows of this weight matrix
  int tile_begin;         // first m-tile of the segment
  int out_col;            // EPI_STORE_F32: column offset of this segment in the output row
  int n_kb_pack;          // packed: 128-byte K boxes per 128-row tile
  const uint8_t *packed;  // packed image of this matrix (see PackedLayout), or null
};

// EPI_QKV: the Q/K/V product's epilogue post-processes the heads (plain head RMSNorm and
// split-half RoPE of query and key heads, a copy of value heads; results in the config
// dtype) and scatters them to the attention's inputs.  Token columns < T are block rows:
// queries token-major [T][Hq*D] (times q_scale unless 0), keys and values [B][Hkv][W][D]
// (each with a bf16 lo plane when the offset is set).  Columns T .. T+n_pend-1 are pending
// context rows (request, position per row) whose keys and values go to the rings when the
// position is live.  Tiles of 128 rows hold 128 / D heads (D = 64 or 128).
struct QkvPost {
  int D, W, n_q_heads, n_kv_heads, T, n_pend, out_f32;
  int n_req, min_back, cap;
  float eps, q_scale;
  const float2 *rope;           // [token][D/2] (cos, sin) by token column
  const void *q_norm, *k_norm;  // [D] head-norm gains
  void *q, *kblk, *vblk;
  size_t q_lo, kv_lo;           // element offsets of the lo planes (0: none)
  void *kring, *vring;          // [B][Hkv][cap][D]
  const int32_t *row_req;       // [n_pend]
  const int64_t *row_pos, *frontier;
};

struct __align__(16) GemmArgs {
  int K, n_tokens, block_n, n_tiles_n, m_tiles, kb, n_ctas, n_segs, stages, pair_mode;
  int kbox;                       // 128-byte-wide K boxes per pipeline stage (1, 2 or 4)
  // Split activations: the activation operand is a bf16 pair x = hi + lo stored as two
  // row blocks [hi rows; lo rows] (lo block starting at row lo_row).  The MMA runs on
  // block_n = 2 * ln columns (ln = logical tokens of a tile) and the epilogue adds the
  // two halves, so activations enter at ~16-bit instead of 8-bit mantissa precision
  // while the weight tile is still read once.
  int split, ln, lo_row;
  int packed;                     // weights come from packed images (contiguous bulk copies)
  long long units;
  int grain;                      // units per scheduling grain (1, or kb: whole tiles per CTA)
  int epi;
  int ld_out, ld_act, block_w, vocab;
  long long act_lo;               // SWIGLU: element offset of the lo block of out_act (0: none)
  float *out_f32;
  const float *row_scale;
  void *out_act;
  float *amax_val;                // [m_tiles][n_tokens]
  int32_t *amax_idx;
  float *topk_val;                // [m_tiles][n_tokens][kTopK], descending
  int32_t *topk_idx;
  const float *wscale;            // TOPK: per weight row score scale (FP8 row scales), or null
  float *partials;                // [n_ctas][2][block_n * 128] fp32 stream-K partial tiles
  unsigned *counters;             // [2][n_counter_tiles] arrival / done counters (start at 0)
  int n_counter_tiles;
  QkvPost qkv;                    // EPI_QKV
  GemmSeg seg[kMaxSegs];
};

struct GemmMaps {
  CUtensorMap a[kMaxSegs];    // weight maps (pair mode: a[0] gate, a[1] up, 64-row boxes)
  CUtensorMap b;              // activation map [n_tokens, K]
  CUtensorMap out[kMaxSegs];  // result maps [n_tokens, rows], boxes of 16 tokens: STORE one
                              // per segment, RESID/INJECT out[0] = x, SWIGLU out[0] with the
                              // hi and lo planes as a third dimension
};

// Host description of one GEMM launch.
struct GemmWeight {
  const void *ptr;
  int rows;
  const void *packed;  // packed image of the matrix (pair mode: the interleaved pair), or null
};
// Operand element type of a GEMM: bf16, fp32 (tf32 products), FP8 e4m3 (both operands one
// byte per element; packed weights only) or fp16 (packed weights converted from bf16).
enum GemmType : int { GT_BF16 = 0, GT_F32 = 1, GT_E4M3 = 2, GT_F16 = 3 };
struct Fp8E4M3 {
  uint8_t bits;
};
struct GemmPlan {
  int dtype;                 // GemmType
  int K;
  int n_tokens;
  const void *x;             // activations [n_tokens, K] (config dtype), dev
  int n_w;
  GemmWeight w[kMaxSegs];
  bool pair_mode;            // SwiGLU: w[0] = gate, w[1] = up (same rows)
  bool split;                // x is a hi/lo pair [2][round_up(n_tokens,16)][K] (bf16 only)
  GemmArgs args;             // epilogue fields filled by the caller; layout by the launcher
};

// Stream-K scratch a GEMM launch may use.
struct GemmScratch {
  float *partials;
  size_t partial_floats;
  unsigned *counters;  // 2 * n_counters words, zero on entry; every launch leaves them zero
  size_t n_counters;   // tiles a launch may have
};

unsigned take_error_word_gemm();
unsigned take_error_word_att();
unsigned take_error_word_small();
unsigned take_error_word_head8();
unsigned take_error_word_bridge();

// ------------------------------------------------------------------ packed weights
// Packed image of one [rows, K] matrix: 128-row tiles, each split into 128-byte K boxes;
// box (tile t, box k) is 16 KB at ((t * n_kb) + k) * 16384, in the 128-byte-swizzled
// shared-memory order (16-byte chunk c of row r stored at chunk c ^ (r % 8)).  A pair
// image (SwiGLU gate/up) has tiles of 64 gate rows followed by the same 64 up rows.
constexpr size_t kPackBox = 16384;
inline size_t packed_kb(int K, int elem) { return (static_cast<size_t>(K) * elem + 127) / 128; }
inline size_t packed_matrix_bytes(int rows, int K, int elem, bool pair) {
  const size_t rt = pair ? (static_cast<size_t>(rows) + 63) / 64 : (static_cast<size_t>(rows) + 127) / 128;
  return rt * packed_kb(K, elem) * kPackBox;
}
struct PackedLayout {
  size_t w_feature, head, g_recv, g_pred, a_val;
  size_t wq[BD_MAX_LAYERS], wk[BD_MAX_LAYERS], wv[BD_MAX_LAYERS], wo[BD_MAX_LAYERS];
  size_t gate_up[BD_MAX_LAYERS], w_down[BD_MAX_LAYERS], r_read[BD_MAX_LAYERS],
      w_write[BD_MAX_LAYERS], conv_a[BD_MAX_LAYERS], conv_m[BD_MAX_LAYERS];
  size_t total;
};
PackedLayout packed_layout(const bd_config *c);
// Empty when the configuration passes the checks every entry point applies.
std::string validate_config(const bd_config *c);
// In a bf16 config the packed image stores the attention-branch matrices (W_q, W_k, W_v,
// W_o and the attention branch's convolution delta), the MLP matrices (gate/up, down, and
// the MLP branch's convolution delta) and the head as fp16: those products take fp16
// activations (one operand of 11 significant bits instead of a bf16 hi+lo pair), which
// halves their tensor work, activation traffic and shared memory per stage.  W_feature and
// the bridge matrices stay bf16.
inline bool packed_f16(const bd_config *c) { return c->dtype == BD_BF16; }
std::string pack_all(const bd_config *c, const bd_weights *w, uint8_t *base, cudaStream_t s);
unsigned take_error_word_pack();

size_t gemm_partial_floats(int n_ctas, int block_n);
// 2-D tiled tensor map of a row-major [outer, inner] matrix (rows `stride` elements apart,
// 0 = inner) with boxes of box_outer x box_inner elements, 128-byte swizzled when
// `swizzle`; out-of-bounds elements read as zero.  Encoded once per distinct argument set.
std::string make_tensor_map_2d(CUtensorMap *out, const void *ptr, int dtype, int inner, int outer,
                               int box_inner, int box_outer, bool swizzle, long long stride = 0);
int num_sms();
int gemm_block_n(int n_tokens);
// Upper bound on the token tiles of a GEMM over n_tokens, whatever tile width it takes.
int gemm_max_n_tiles(int n_tokens);

// Launch; returns an error message or empty string.
std::string launch_gemm(GemmPlan &plan, const GemmScratch &scratch, cudaStream_t stream);

// ------------------------------------------------------------------ launch helper
// Launch with programmatic stream serialisation (PDL) so the next kernel's prologue can
// overlap this kernel's tail; every kernel calls pdl_wait() before dependent accesses.
void count_launch();
void set_last_error(const std::string &msg);

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launch();
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The same launch as a cluster of cluster_x consecutive CTAs along x (cluster_x divides
// grid.x); cluster_x = 1 is a plain launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t stream, int cluster_x, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(cluster_x);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  count_launch();
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace bd
