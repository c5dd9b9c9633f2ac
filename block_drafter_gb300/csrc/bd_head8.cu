// FP8 retrieval head ("DSpine for Qwen3.8-27B: Causal Features Through Depth", section "The
// last write is refined using discrete candidates": the optimized path scores the whole
// vocabulary with a row-scaled FP8 copy of the head, keeps 128 candidates, rescores them
// with the BF16 head and keeps 16).
//
//   head image   every vocabulary row v coded as e4m3(E_v / s_v), s_v = max|E_v| / 448, in
//                the packed 128-row x 128-byte box layout of the tensor-core GEMM, then the
//                fp32 scales s_v
//   hidden code  the same row-scaled code of each hidden row (its scale is common to the
//                row's scores and is not applied)
//   retrieval    an e4m3 x e4m3 tcgen05 GEMM (kind::f8f6f4) whose epilogue keeps each
//                128-row tile's 16 best s_v * (q_v . q_h) per row
//   selection    the n_cand best of those per row: radix selection of the n_cand-th
//                largest score, equal scores to the lower id
//   rescoring    exact BF16 dot products of the candidates, then the k best
#include "bd_device.cuh"
#include "bd_internal.h"
#include "bd_kernels.h"

namespace bd {

BD_DEFINE_ERROR_TAKER(take_error_word_head8)

constexpr float kE4M3Max = 448.f;

static std::string err(const char *what, cudaError_t e) {
  return e == cudaSuccess ? std::string() : std::string(what) + ": " + cudaGetErrorString(e);
}

// 16 consecutive fp32 values as 16 e4m3 codes (byte j = value j).
__device__ __forceinline__ uint4 code16(const float (&x)[16], float s) {
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t lo = e4m3x2(__fdiv_rn(x[4 * q + 0], s), __fdiv_rn(x[4 * q + 1], s));
    const uint32_t hi = e4m3x2(__fdiv_rn(x[4 * q + 2], s), __fdiv_rn(x[4 * q + 3], s));
    w[q] = lo | (hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Row scale max|row| / 448 (1 for an all-zero row, whose codes are all zero).
__device__ __forceinline__ float fp8_scale(float mx) {
  const float s = __fdiv_rn(mx, kE4M3Max);
  return s > 0.f ? s : 1.f;
}

// One CTA per 128-row tile of the head: the tile's row scales, then every 16 KB K box of
// the tile in the 128-byte-swizzled order (16-byte chunk c of row r at chunk c ^ (r % 8)).
__global__ void __launch_bounds__(256) head_fp8_pack_kernel(const __nv_bfloat16 *E, int V, int H,
                                                            int n_kb, uint8_t *img, float *scales) {
  __shared__ float s_row[128];
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = warp; r < 128; r += 8) {
    const int v = t * 128 + r;
    float mx = 0.f;
    if (v < V) {
      const __nv_bfloat16 *row = E + static_cast<size_t>(v) * H;
      for (int j = lane * 8; j < H; j += 256) {
        const uint4 u = *reinterpret_cast<const uint4 *>(row + j);
        const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(p2[e]);
          mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
      }
    }
    mx = warp_max(mx);
    if (lane == 0) {
      const float s = fp8_scale(mx);
      s_row[r] = s;
      if (v < V) scales[v] = s;
    }
  }
  __syncthreads();
  for (int kbx = 0; kbx < n_kb; ++kbx) {
    uint8_t *out = img + (static_cast<size_t>(t) * n_kb + kbx) * kPackBox;
    for (int q = threadIdx.x; q < 1024; q += blockDim.x) {
      const int r = q >> 3, c = q & 7;
      const int v = t * 128 + r, col = kbx * 128 + c * 16;
      uint4 code = make_uint4(0u, 0u, 0u, 0u);
      if (v < V && col < H) {
        float x[16];
        const __nv_bfloat16 *src = E + static_cast<size_t>(v) * H + col;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint4 u = *reinterpret_cast<const uint4 *>(src + 8 * h);
          const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(p2[e]);
            x[8 * h + 2 * e] = f.x;
            x[8 * h + 2 * e + 1] = f.y;
          }
        }
        code = code16(x, s_row[r]);
      }
      *reinterpret_cast<uint4 *>(out + r * 128 + ((c ^ (r & 7)) << 4)) = code;
    }
  }
}

// One CTA per hidden row: its row-scaled e4m3 code [H] (H a multiple of 16).
__global__ void __launch_bounds__(256) code_rows_kernel(const float *h, int H, uint8_t *q,
                                                        ZeroSpan z) {
  __shared__ float red[8];
  pdl_wait();
  pdl_trigger();
  zero_span(z);
  const int row = blockIdx.x;
  const float *x = h + static_cast<size_t>(row) * H;
  float mx = 0.f;
  for (int j = threadIdx.x * 4; j < H; j += blockDim.x * 4) {
    const float4 f = *reinterpret_cast<const float4 *>(x + j);
    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w))));
  }
  mx = warp_max(mx);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = 0.f;
  for (int i = 0; i < 8; ++i) mx = fmaxf(mx, red[i]);
  const float s = fp8_scale(mx);
  for (int j = threadIdx.x * 16; j < H; j += blockDim.x * 16) {
    float v[16];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float4 f = *reinterpret_cast<const float4 *>(x + j + 4 * e);
      v[4 * e] = f.x;
      v[4 * e + 1] = f.y;
      v[4 * e + 2] = f.z;
      v[4 * e + 3] = f.w;
    }
    *reinterpret_cast<uint4 *>(q + static_cast<size_t>(row) * H + j) = code16(v, s);
  }
}

// Order-preserving map of a float to an unsigned key (larger float, larger key).
__device__ __forceinline__ uint32_t fkey(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One CTA (1024 threads) per row: the n_cand best of the row's per-tile candidate lists
// val/idx [m_tiles][rows][kTopK].  The n_cand-th largest score is found by four 8-bit
// radix passes over the keys held in shared memory; every candidate above it is taken,
// and of those equal to it the ones with the lowest ids (tie buffer `ties` [rows][N]).
// The selection is written unordered to cand [rows][n_cand].
__global__ void __launch_bounds__(1024) select_cand_kernel(const float *val, const int32_t *idx,
                                                           int m_tiles, int rows, int n_cand,
                                                           int32_t *ties, int32_t *cand) {
  extern __shared__ uint32_t keys[];  // [N], then the per-warp histograms [32][256]
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_prefix, s_need, s_n_gt, s_n_tie;
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x, tid = threadIdx.x;
  const int N = m_tiles * kTopK;
  auto src = [&](int p) { return (static_cast<size_t>(p / kTopK) * rows + row) * kTopK + p % kTopK; };
#pragma unroll 4
  for (int p = tid; p < N; p += blockDim.x) keys[p] = fkey(val[src(p)]);
  if (tid == 0) {
    s_prefix = 0u;
    s_need = static_cast<uint32_t>(n_cand);
    s_n_gt = 0u;
    s_n_tie = 0u;
  }
  // The scores of a row crowd into few digits, so each warp counts into its own histogram
  // (same-address atomics then only collide within a warp) and the 32 are summed.
  uint32_t *whist = keys + N + ((tid >> 5) << 8);
  uint32_t mask = 0u;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int d = tid; d < 32 * 256; d += blockDim.x) keys[N + d] = 0u;
    __syncthreads();
    const uint32_t prefix = s_prefix;
    for (int p = tid; p < N; p += blockDim.x)
      if ((keys[p] & mask) == prefix) atomicAdd(&whist[(keys[p] >> shift) & 255u], 1u);
    __syncthreads();
    for (int d = tid; d < 256; d += blockDim.x) {
      uint32_t t = 0u;
#pragma unroll 8
      for (int w = 0; w < 32; ++w) t += keys[N + w * 256 + d];
      hist[d] = t;
    }
    __syncthreads();
    if (tid < 32) {  // the digit holding the need-th largest key, counting from the top
      // lane l owns digits 255 - 8l .. 248 - 8l; an inclusive scan of the lanes' counts
      // gives how many keys lie above each lane's range
      const uint32_t need = s_need;
      uint32_t own = 0u;
#pragma unroll
      for (int e = 0; e < 8; ++e) own += hist[255 - 8 * tid - e];
      uint32_t incl = own;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
        if (tid >= off) incl += o;
      }
      const uint32_t above = incl - own;
      if (above < need && incl >= need) {  // exactly one lane
        uint32_t cum = above;
        int d = 255 - 8 * tid;
        for (int e = 0; e < 7; ++e, --d) {
          if (cum + hist[d] >= need) break;
          cum += hist[d];
        }
        s_need = need - cum;
        s_prefix = prefix | (static_cast<uint32_t>(d) << shift);
      }
    }
    mask |= 255u << shift;
    __syncthreads();
  }
  const uint32_t T = s_prefix;
  const uint32_t need_eq = s_need;  // keys equal to T still to take
  int32_t *out = cand + static_cast<size_t>(row) * n_cand;
  int32_t *tie = ties + static_cast<size_t>(row) * N;
  for (int p = tid; p < N; p += blockDim.x) {
    if (keys[p] > T) {
      out[atomicAdd(&s_n_gt, 1u)] = idx[src(p)];
    } else if (keys[p] == T) {
      tie[atomicAdd(&s_n_tie, 1u)] = idx[src(p)];
    }
  }
  __syncthreads();
  const uint32_t n_gt = s_n_gt, n_tie = s_n_tie;
  if (n_gt + need_eq != static_cast<uint32_t>(n_cand)) {  // cannot happen; keep the output sane
    if (tid == 0) atomicOr(&g_error_word, DEVERR_BAD_INDEX);
    return;
  }
  // the need_eq lowest ids among the ties: each tie's rank among them (ids are distinct)
  for (uint32_t i = tid; i < n_tie; i += blockDim.x) {
    const int id = tie[i];
    uint32_t rank = 0u;
    for (uint32_t j = 0; j < n_tie && rank < need_eq; ++j) rank += tie[j] < id ? 1u : 0u;
    if (rank < need_eq) out[n_gt + rank] = id;
  }
}

// Exact scores E[cand] . h of the candidates (bf16 head rows, fp32 hidden row, fp32 sums):
// CTA (g, row) of 512 threads scores candidates 16 g .. 16 g + 15 of the row, one warp
// each, into scores [rows][n_cand].  The row's last CTA to finish (a per-row counter,
// cleared again by that CTA) then takes the k best in candidate order.
__global__ void __launch_bounds__(512) rescore_kernel(const __nv_bfloat16 *E, int V, int H,
                                                      const float *hidden, const int32_t *cand,
                                                      int n_cand, int k, float *scores,
                                                      unsigned *row_done, int32_t *tok_out,
                                                      float *score_out) {
  __shared__ unsigned s_last;
  pdl_wait();
  pdl_trigger();
  const int g = blockIdx.x, row = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t *cr = cand + static_cast<size_t>(row) * n_cand;
  float *sr = scores + static_cast<size_t>(row) * n_cand;
  const int c = g * 16 + warp;
  if (c < n_cand) {
    int id = cr[c];
    if (id < 0 || id >= V) {
      if (lane == 0) atomicOr(&g_error_word, DEVERR_BAD_INDEX);
      id = 0;
    }
    const __nv_bfloat16 *e = E + static_cast<size_t>(id) * H;
    const float *x = hidden + static_cast<size_t>(row) * H;
    float acc = 0.f;
#pragma unroll 5
    for (int j = lane * 8; j < H; j += 256) {
      const uint4 u = *reinterpret_cast<const uint4 *>(e + j);
      const float4 x0 = *reinterpret_cast<const float4 *>(x + j);
      const float4 x1 = *reinterpret_cast<const float4 *>(x + j + 4);
      const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
      const float2 f0 = __bfloat1622float2(p2[0]), f1 = __bfloat1622float2(p2[1]);
      const float2 f2 = __bfloat1622float2(p2[2]), f3 = __bfloat1622float2(p2[3]);
      acc = fmaf(f0.x, x0.x, acc);
      acc = fmaf(f0.y, x0.y, acc);
      acc = fmaf(f1.x, x0.z, acc);
      acc = fmaf(f1.y, x0.w, acc);
      acc = fmaf(f2.x, x1.x, acc);
      acc = fmaf(f2.y, x1.y, acc);
      acc = fmaf(f3.x, x1.z, acc);
      acc = fmaf(f3.y, x1.w, acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) sr[c] = acc;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&row_done[row], 1u) == gridDim.x - 1 ? 1u : 0u;
  __syncthreads();
  if (!s_last || warp != 0) return;
  __threadfence();
  if (lane == 0) row_done[row] = 0u;  // ready for the next call
  // each lane keeps its (up to 8) candidates sorted; k rounds of a warp-wide best
  constexpr int kPer = 8;
  float lv[kPer];
  int li[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int cc = lane + 32 * i;
    lv[i] = cc < n_cand ? __ldcg(sr + cc) : -INFINITY;
    li[i] = cc < n_cand ? cr[cc] : 0x7fffffff;
  }
#pragma unroll
  for (int i = 1; i < kPer; ++i)
#pragma unroll
    for (int j = i; j > 0; --j)
      if (cand_better(lv[j], li[j], lv[j - 1], li[j - 1])) {
        const float tv = lv[j];
        lv[j] = lv[j - 1];
        lv[j - 1] = tv;
        const int ti = li[j];
        li[j] = li[j - 1];
        li[j - 1] = ti;
      }
  for (int r = 0; r < k; ++r) {
    float bv = lv[0];
    int bi = li[0];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (cand_better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (li[0] == bi) {
#pragma unroll
      for (int i = 0; i < kPer - 1; ++i) {
        lv[i] = lv[i + 1];
        li[i] = li[i + 1];
      }
      lv[kPer - 1] = -INFINITY;
      li[kPer - 1] = 0x7fffffff;
    }
    if (lane == 0) {
      tok_out[static_cast<size_t>(row) * k + r] = bi;
      if (score_out) score_out[static_cast<size_t>(row) * k + r] = bv;
    }
  }
}

// ------------------------------------------------------------------ host
size_t head_fp8_image_bytes(int V, int H) {
  return ((static_cast<size_t>(V) + 127) / 128) * packed_kb(H, 1) * kPackBox;
}

std::string launch_head_fp8_pack(const void *E, int V, int H, void *img, cudaStream_t s) {
  const int tiles = (V + 127) / 128;
  const int n_kb = static_cast<int>(packed_kb(H, 1));
  uint8_t *base = static_cast<uint8_t *>(img);
  float *scales = reinterpret_cast<float *>(base + head_fp8_image_bytes(V, H));
  return err("fp8 head pack", launch_pdl(head_fp8_pack_kernel, dim3(tiles), dim3(256), 0, s,
                                         static_cast<const __nv_bfloat16 *>(E), V, H, n_kb, base,
                                         scales));
}

std::string launch_code_rows(const float *h, int rows, int H, void *q, ZeroSpan z, cudaStream_t s) {
  return err("fp8 code rows", launch_pdl(code_rows_kernel, dim3(rows), dim3(256), 0, s, h, H,
                                         static_cast<uint8_t *>(q), z));
}

size_t select_cand_smem(int m_tiles) {
  return (static_cast<size_t>(m_tiles) * kTopK + 32 * 256) * sizeof(uint32_t);
}

std::string launch_select_cand(const float *val, const int32_t *idx, int m_tiles, int rows,
                               int n_cand, int32_t *ties, int32_t *cand, cudaStream_t s) {
  const size_t smem = select_cand_smem(m_tiles);
  static size_t set_to = 0;
  if (smem > 48 * 1024 && smem > set_to) {
    cudaError_t e = cudaFuncSetAttribute(select_cand_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return err("fp8 candidate selection", e);
    set_to = smem;
  }
  return err("fp8 candidate selection",
             launch_pdl(select_cand_kernel, dim3(rows), dim3(1024), smem, s, val, idx, m_tiles,
                        rows, n_cand, ties, cand));
}

std::string launch_rescore(const void *E, int V, int H, const float *hidden, const int32_t *cand,
                           int rows, int n_cand, int k, float *scores, unsigned *row_done,
                           int32_t *tok_out, float *score_out, cudaStream_t s) {
  return err("fp8 rescoring",
             launch_pdl(rescore_kernel, dim3((n_cand + 15) / 16, rows), dim3(512), 0, s,
                        static_cast<const __nv_bfloat16 *>(E), V, H, hidden, cand, n_cand, k,
                        scores, row_done, tok_out, score_out));
}

}  // namespace bd
