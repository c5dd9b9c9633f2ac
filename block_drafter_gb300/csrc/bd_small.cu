// Small bandwidth-trivial kernels around the GEMMs: embedding gather and RoPE tables,
// row norms, the DSpine code finalisation and gated message, the split-vocab argmax
// reduction.  Each launches with programmatic dependent launch and waits for the
// previous kernel before touching data it produced or consumes.
#include "bd_device.cuh"

#include <type_traits>
#include "bd_internal.h"
#include "bd_kernels.h"

namespace bd {

BD_DEFINE_ERROR_TAKER(take_error_word_small)

__device__ __forceinline__ float block_sum(float v, float *red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float s = 0.f;
  for (int i = 0; i < nw; ++i) s += red[i];
  return s;
}

// (cos, sin) of pos * inv_freq[j]: the product and its reduction modulo 2 pi are done in
// double precision so that large positions keep full single-precision angles.  The
// multiple of 2 pi comes from a product with 1 / (2 pi) (a rounding there can leave the
// reduced angle just outside [0, 2 pi), which sincosf takes as it is).
__device__ __forceinline__ float2 rope_cs(long long pos, double inv) {
  const double two_pi = 6.283185307179586476925286766559;
  const double inv_two_pi = 0.15915494309189533576888376337251;
  double ang = static_cast<double>(pos) * inv;
  ang -= floor(ang * inv_two_pi) * two_pi;
  float s, c;
  sincosf(static_cast<float>(ang), &s, &c);
  return make_float2(c, s);
}


template <typename T> __device__ __forceinline__ float4 load4(const T *p, int i4);
template <> __device__ __forceinline__ float4 load4<float>(const float *p, int i4) {
  return reinterpret_cast<const float4 *>(p)[i4];
}
template <> __device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16 *p, int i4) {
  const uint2 u = reinterpret_cast<const uint2 *>(p)[i4];
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&u.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&u.y);
  const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}
template <typename T>
__global__ void round_prep_kernel(const T *embed, int H, int V, const int32_t *anchors,
                                  const int64_t *frontier, int W, int n_tok, int mask_id, float *x,
                                  float2 *rope, int half, RopeFreq freq, const int64_t *pend_pos,
                                  ZeroSpan z) {
  const int tok = blockIdx.x, b = tok / W, i = tok % W;
  pdl_wait();
  pdl_trigger();
  zero_span(z);
  if (tok >= n_tok) {  // a pending context row: its RoPE row only
    const long long pos = pend_pos[tok - n_tok];
    for (int j = threadIdx.x; j < half; j += blockDim.x)
      rope[static_cast<size_t>(tok) * half + j] = rope_cs(pos, freq.inv[j]);
    return;
  }
  int id = i == 0 ? anchors[b] : mask_id;
  if (id < 0 || id >= V) {
    if (threadIdx.x == 0) atomicOr(&g_error_word, DEVERR_BAD_INDEX);
    id = 0;
  }
  const T *e = embed + static_cast<size_t>(id) * H;
  float *xr = x + static_cast<size_t>(tok) * H;
  constexpr int U = 8;  // float4 loads in flight per thread (H % 4 == 0)
  for (int base = threadIdx.x; base < H / 4; base += U * blockDim.x) {
    float4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i4 = base + u * blockDim.x;
      v[u] = i4 < H / 4 ? load4<T>(e, i4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i4 = base + u * blockDim.x;
      if (i4 < H / 4) reinterpret_cast<float4 *>(xr)[i4] = v[u];
    }
  }
  const long long pos = frontier[b] + i;
  for (int j = threadIdx.x; j < half; j += blockDim.x)
    rope[static_cast<size_t>(tok) * half + j] = rope_cs(pos, freq.inv[j]);
}

__global__ void rope_table_kernel(const int64_t *pos, int n, float2 *rope, int half,
                                  RopeFreq freq, ZeroSpan z) {
  pdl_wait();
  pdl_trigger();
  zero_span(z);
  const int total = n * half;
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < total; t += gridDim.x * blockDim.x) {
    const int r = t / half, j = t % half;
    rope[t] = rope_cs(pos[r], freq.inv[j]);
  }
}

template <typename T> __device__ __forceinline__ void store4(T *p, int i4, float4 v);
template <> __device__ __forceinline__ void store4<__half>(__half *p, int i4, float4 v) {
  flag_f16_range(f16_out_of_range(v.x) || f16_out_of_range(v.y) || f16_out_of_range(v.z) ||
                 f16_out_of_range(v.w));
  __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t *>(&a);
  u.y = *reinterpret_cast<uint32_t *>(&b);
  reinterpret_cast<uint2 *>(p)[i4] = u;
}
template <> __device__ __forceinline__ void store4<float>(float *p, int i4, float4 v) {
  reinterpret_cast<float4 *>(p)[i4] = v;
}
template <> __device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16 *p, int i4, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t *>(&a);
  u.y = *reinterpret_cast<uint32_t *>(&b);
  reinterpret_cast<uint2 *>(p)[i4] = u;
}

// One CTA per row.  Rows up to kNormVec * 4 * blockDim elements stay in registers between
// the sum-of-squares and the output pass (float4 loads, all issued before the reduction).
constexpr int kNormVec = 8;

// DFlash2 grouped convolution of one block row (channels 4*i4 .. 4*i4+3, one group since
// the group width is a multiple of 4): (base[side,0] + delta[row,side,0,g]) * X[row]
// + [i >= 1] (base[side,1] + delta[row,side,1,g]) * X[row - 1].  X rows are H wide,
// delta rows hold [2 sides][2 taps][G groups].
template <typename T>
__device__ __forceinline__ float4 conv_row4(const float *X, const float *delta, const T *base,
                                            int H, int gw, int side, int row, bool has_prev, int i4) {
  const int G = H / gw, g = (4 * i4) / gw;
  const float *d = delta + static_cast<size_t>(row) * 4 * G + side * 2 * G;
  const float dc = d[g], dp = d[G + g];
  const float4 bc = load4<T>(base + static_cast<size_t>(side) * 2 * H, i4);
  const float4 x = reinterpret_cast<const float4 *>(X + static_cast<size_t>(row) * H)[i4];
  float4 o = make_float4((bc.x + dc) * x.x, (bc.y + dc) * x.y, (bc.z + dc) * x.z, (bc.w + dc) * x.w);
  if (has_prev) {
    const float4 bp = load4<T>(base + static_cast<size_t>(side) * 2 * H + H, i4);
    const float4 xp = reinterpret_cast<const float4 *>(X + static_cast<size_t>(row - 1) * H)[i4];
    o.x += (bp.x + dp) * xp.x;
    o.y += (bp.y + dp) * xp.y;
    o.z += (bp.z + dp) * xp.z;
    o.w += (bp.w + dp) * xp.w;
  }
  return o;
}

// T: weight (gain, convolution base) type; O: the normalised output's type.
template <typename T, typename O>
__global__ void __launch_bounds__(256) rownorm_kernel(float *x, int H, const T *gain, float eps,
                                                      int mode, O *out, float *r_out,
                                                      float *f32_out, float *head_out, int W,
                                                      size_t lo_off, ConvFinish cf) {
  __shared__ float red[32];
  const int row = blockIdx.x;
  const int H4 = H / 4;
  // the gain (a weight: no earlier kernel writes it) is loaded before the dependency wait
  const bool has_gain = mode != NORM_BRIDGE && gain != nullptr;
  float4 gv[kNormVec];
#pragma unroll
  for (int k = 0; k < kNormVec; ++k) {
    const int i4 = threadIdx.x + k * blockDim.x;
    gv[k] = has_gain && i4 < H4 ? load4<T>(gain, i4) : make_float4(1.f, 1.f, 1.f, 1.f);
  }
  pdl_wait();
  pdl_trigger();
  float *xr = x + static_cast<size_t>(row) * H;
  const bool fin = cf.z != nullptr;
  const bool has_prev = (row % W) != 0;
  // x (+ the branch output's side-1 convolution, written back: the residual update)
  auto load_x = [&](int i4) -> float4 {
    float4 t = reinterpret_cast<const float4 *>(xr)[i4];
    if (fin) {
      const float4 c = conv_row4<T>(cf.z, cf.delta, static_cast<const T *>(cf.base), H, cf.gw, 1,
                                    row, has_prev, i4);
      t = make_float4(t.x + c.x, t.y + c.y, t.z + c.z, t.w + c.w);
      reinterpret_cast<float4 *>(xr)[i4] = t;
    }
    return t;
  };
  float4 xv[kNormVec];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kNormVec; ++k) {
    const int i4 = threadIdx.x + k * blockDim.x;
    xv[k] = i4 < H4 ? load_x(i4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int k = 0; k < kNormVec; ++k)
    ss += xv[k].x * xv[k].x + xv[k].y * xv[k].y + xv[k].z * xv[k].z + xv[k].w * xv[k].w;
  for (int i4 = threadIdx.x + kNormVec * blockDim.x; i4 < H4; i4 += blockDim.x) {
    const float4 t = load_x(i4);  // written back: the output pass re-reads x
    ss += t.x * t.x + t.y * t.y + t.z * t.z + t.w * t.w;
  }
  ss = block_sum(ss, red);
  float scale;
  if (mode == NORM_BRIDGE) {
    const float r = sqrtf(ss / H);
    scale = 1.f / (r + eps);
    if (threadIdx.x == 0) r_out[row] = r;
  } else {
    scale = rsqrtf(ss / H + eps);
  }
  const int i = row % W;
  O *orow = (mode == NORM_FINAL) ? nullptr : out + static_cast<size_t>(row) * H;
  float *hrow = nullptr;
  if (mode == NORM_FINAL && head_out != nullptr && i > 0)
    hrow = head_out + (static_cast<size_t>(row / W) * (W - 1) + (i - 1)) * H;
  float *frow = f32_out ? f32_out + static_cast<size_t>(row) * H : nullptr;
  auto emit = [&](int i4, float4 t, float4 g) {
    float4 y = make_float4(t.x * scale, t.y * scale, t.z * scale, t.w * scale);
    if (mode != NORM_BRIDGE) {
      y.x *= g.x;
      y.y *= g.y;
      y.z *= g.z;
      y.w *= g.w;
    }
    if (orow) {
      store4<O>(orow, i4, y);
      if (lo_off && mode == NORM_CTX) {
        store4<O>(orow + lo_off, i4, make_float4(0.f, 0.f, 0.f, 0.f));
      } else if (lo_off) {  // residual of the rounding: hi + lo carries ~16 mantissa bits
        const float4 h = make_float4(to_f<O>(from_f<O>(y.x)), to_f<O>(from_f<O>(y.y)),
                                     to_f<O>(from_f<O>(y.z)), to_f<O>(from_f<O>(y.w)));
        store4<O>(orow + lo_off, i4, make_float4(y.x - h.x, y.y - h.y, y.z - h.z, y.w - h.w));
      }
    }
    if (hrow) reinterpret_cast<float4 *>(hrow)[i4] = y;
    if (frow) reinterpret_cast<float4 *>(frow)[i4] = y;
  };
#pragma unroll
  for (int k = 0; k < kNormVec; ++k) {
    const int i4 = threadIdx.x + k * blockDim.x;
    if (i4 < H4) emit(i4, xv[k], gv[k]);
  }
  for (int i4 = threadIdx.x + kNormVec * blockDim.x; i4 < H4; i4 += blockDim.x)
    emit(i4, reinterpret_cast<const float4 *>(xr)[i4],
         has_gain ? load4<T>(gain, i4) : make_float4(1.f, 1.f, 1.f, 1.f));
}

template <typename T>
__device__ __forceinline__ void store_split(T *p, size_t i, size_t lo_off, float v) {
  if (std::is_same<T, __half>::value) flag_f16_range(f16_out_of_range(v));
  const T h = from_f<T>(v);
  p[i] = h;
  if (lo_off) p[lo_off + i] = from_f<T>(v - to_f<T>(h));
}

// DFlash2 branch input: out[row] = Conv_0(X)[row] (the side-0 convolution of the
// normalised branch input), as a split pair when lo_off != 0.  One CTA per block row.
template <typename T, typename O>
__global__ void __launch_bounds__(256) conv_prepare_kernel(const float *X, const float *delta,
                                                           const T *base, int H, int gw, int W,
                                                           O *out, size_t lo_off) {
  const int row = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  const bool has_prev = (row % W) != 0;
  O *o = out + static_cast<size_t>(row) * H;
  for (int i4 = threadIdx.x; i4 < H / 4; i4 += blockDim.x) {
    const float4 y = conv_row4<T>(X, delta, base, H, gw, 0, row, has_prev, i4);
    store4<O>(o, i4, y);
    if (lo_off) {
      const float4 h = make_float4(to_f<O>(from_f<O>(y.x)), to_f<O>(from_f<O>(y.y)),
                                   to_f<O>(from_f<O>(y.z)), to_f<O>(from_f<O>(y.w)));
      store4<O>(o + lo_off, i4, make_float4(y.x - h.x, y.y - h.y, y.z - h.z, y.w - h.w));
    }
  }
}

// One warp per (row, head).  Lane l holds elements [l*E, l*E + E) of the head (E = D/32);
// the split-half RoPE partner of element d is d +- D/2, which lives in lane l ^ 16.
template <typename T, int E>
__global__ void __launch_bounds__(256) head_post_kernel(const __grid_constant__ HeadPostArgs a) {
  const int warp = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int rr = warp / a.total_heads;  // context row
  int hg = warp % a.total_heads;
  const bool live = rr < a.rows;
  int si = 0;
  while (si + 1 < a.n_segs && hg >= a.seg[si].n_heads) {
    hg -= a.seg[si].n_heads;
    ++si;
  }
  const HeadSeg sg = a.seg[si];
  const int D = E * 32, half = D / 2;
  const int d0 = lane * E;
  // the head-norm gain (a weight: no earlier kernel writes it) before the dependency wait
  float gn[E];
#pragma unroll
  for (int e = 0; e < E; ++e)
    gn[e] = live && sg.kind == HK_K ? to_f<T>(static_cast<const T *>(sg.norm)[d0 + e]) : 1.f;
  pdl_wait();
  pdl_trigger();
  if (!live) return;
  const float *src = a.raw + static_cast<size_t>(rr) * a.ld_raw + sg.col0 + hg * D + d0;
  float v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = src[e];
  if (sg.kind == HK_K) {
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) ss += v[e] * v[e];
    ss = warp_sum(ss);
    const float inv = rsqrtf(ss / static_cast<float>(D) + a.eps);
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] *= inv * gn[e];
    const float2 *cs = a.rope + static_cast<size_t>(rr) * half;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float pv = __shfl_xor_sync(0xffffffffu, v[e], 16);
      const int d = d0 + e;
      const float2 c = cs[d % half];
      v[e] = d < half ? v[e] * c.x - pv * c.y : v[e] * c.x + pv * c.y;
    }
  }
  const int req = a.row_req[rr];
  const long long pos = a.row_pos[rr];
  if (req < 0 || req >= a.n_req || pos < 0) {
    if (lane == 0) atomicOr(&g_error_word, DEVERR_BAD_INDEX);
    return;
  }
  const long long F = a.frontier[req];
  if (a.min_back > 0 && (pos < F - a.min_back || pos >= F)) {
    if (lane == 0) atomicOr(&g_error_word, DEVERR_BAD_INDEX);
    return;
  }
  if (pos < F - sg.cap || pos >= F) return;  // outside the final live window
  T *dst = static_cast<T *>(sg.dst) +
           ((static_cast<size_t>(req) * a.n_kv_heads + hg) * sg.cap + pos % sg.cap) * D + d0;
#pragma unroll
  for (int e = 0; e < E; ++e) store_split(dst, e, 0, v[e]);
}

template <typename T, typename O>
__global__ void code_kernel(const float *z, int Rc, const T *codebook, const int32_t *anchors,
                            int V, int W, float eps, O *c_out, size_t lo_off) {
  __shared__ float red[32];
  const int row = blockIdx.x, b = row / W, i = row % W;
  pdl_wait();
  pdl_trigger();
  const float scale = sqrtf(static_cast<float>(Rc));
  O *c = c_out + static_cast<size_t>(row) * Rc;
  if (i == 0) {
    int a = anchors[b];
    if (a < 0 || a >= V) {
      if (threadIdx.x == 0) atomicOr(&g_error_word, DEVERR_BAD_INDEX);
      a = 0;
    }
    const T *cb = codebook + static_cast<size_t>(a) * Rc;
    for (int k = threadIdx.x; k < Rc; k += blockDim.x) store_split(c, k, lo_off, scale * to_f<T>(cb[k]));
    return;
  }
  const float *zr = z + static_cast<size_t>(row) * Rc;
  float ss = 0.f;
  for (int k = threadIdx.x; k < Rc; k += blockDim.x) ss += zr[k] * zr[k];
  ss = block_sum(ss, red);
  const float s = scale / (sqrtf(ss) + eps);
  for (int k = threadIdx.x; k < Rc; k += blockDim.x) store_split(c, k, lo_off, zr[k] * s);
}

template <typename T, typename O>
__global__ void message_kernel(const float *pre, int Mc, const T *bias, int W, O *m_out,
                               size_t lo_off) {
  const int row = blockIdx.x, i = row % W;
  pdl_wait();
  pdl_trigger();
  O *m = m_out + static_cast<size_t>(row) * Mc;
  if (i == 0) {
    for (int k = threadIdx.x; k < Mc; k += blockDim.x) store_split(m, k, lo_off, 0.f);
    return;
  }
  const float *recv = pre + static_cast<size_t>(row) * 3 * Mc;         // G c_i
  const float *pred = pre + static_cast<size_t>(row - 1) * 3 * Mc;     // [., G_p c_{i-1}, A c_{i-1}]
  for (int k = threadIdx.x; k < Mc; k += blockDim.x) {
    const float z = recv[k] + pred[Mc + k] + (bias ? to_f<T>(bias[k]) : 0.f);
    const float g = 1.f / (1.f + expf(-z));
    store_split(m, k, lo_off, g * pred[2 * Mc + k]);
  }
}

__global__ void argmax_reduce_kernel(const float *val, const int32_t *idx, int m_tiles, int rows,
                                     int32_t *tok_out, float *max_out) {
  __shared__ float sv[32];
  __shared__ int si[32];
  const int row = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  float best = -INFINITY;
  int bi = 0x7fffffff;
  for (int t = threadIdx.x; t < m_tiles; t += blockDim.x) {
    const float v = val[static_cast<size_t>(t) * rows + row];
    const int i = idx[static_cast<size_t>(t) * rows + row];
    if (v > best || (v == best && i < bi)) {
      best = v;
      bi = i;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > best || (ov == best && oi < bi)) {
      best = ov;
      bi = oi;
    }
  }
  if ((threadIdx.x & 31) == 0) {
    sv[threadIdx.x >> 5] = best;
    si[threadIdx.x >> 5] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    best = sv[0];
    bi = si[0];
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w)
      if (sv[w] > best || (sv[w] == best && si[w] < bi)) {
        best = sv[w];
        bi = si[w];
      }
    tok_out[row] = bi;
    if (max_out) max_out[row] = best;
  }
}

// Candidate order: higher score first, equal scores to the lower id.
// Insert (x, xi) into the sorted list (L, I) of kTopK entries if it beats the last one.
__device__ __forceinline__ bool cand_insert(float (&L)[kTopK], int (&I)[kTopK], float x, int xi) {
  if (!cand_better(x, xi, L[kTopK - 1], I[kTopK - 1])) return false;
  bool placed = false;
#pragma unroll
  for (int j = kTopK - 1; j > 0; --j) {
    if (!placed) {
      if (cand_better(x, xi, L[j - 1], I[j - 1])) {
        L[j] = L[j - 1];
        I[j] = I[j - 1];
      } else {
        L[j] = x;
        I[j] = xi;
        placed = true;
      }
    }
  }
  if (!placed) {
    L[0] = x;
    I[0] = xi;
  }
  return true;
}

// Top-k merge, stage 1: CTA (slice, row) merges the candidate lists of vocabulary tiles
// [slice * per, slice * per + per) of one row into one list.  Each thread inserts the
// lists of its tiles into a private sorted list (a tile's list is sorted, so its scan stops
// at the first candidate that does not enter); the 32 lists of a warp are merged by 16
// rounds of a warp argmax over the list heads (the winner drops its head), then the 8
// warp lists the same way by the first warp.
__global__ void __launch_bounds__(256) topk_slice_kernel(const float *val, const int32_t *idx,
                                                         int m_tiles, int rows, int per,
                                                         float *part_val, int32_t *part_idx) {
  __shared__ float wv[8][kTopK];
  __shared__ int wi[8][kTopK];
  pdl_wait();
  pdl_trigger();
  const int slice = blockIdx.x, row = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float L[kTopK];
  int I[kTopK];
#pragma unroll
  for (int j = 0; j < kTopK; ++j) {
    L[j] = -INFINITY;
    I[j] = 0x7fffffff;
  }
  const int m_end = min(m_tiles, (slice + 1) * per);
  for (int m = slice * per + threadIdx.x; m < m_end; m += blockDim.x) {
    const size_t o = (static_cast<size_t>(m) * rows + row) * kTopK;
    const float4 *pv = reinterpret_cast<const float4 *>(val + o);
    const int4 *pi = reinterpret_cast<const int4 *>(idx + o);
    float4 cv[kTopK / 4];
    int4 ci[kTopK / 4];
#pragma unroll
    for (int q = 0; q < kTopK / 4; ++q) {
      cv[q] = pv[q];
      ci[q] = pi[q];
    }
    const float *fv = reinterpret_cast<const float *>(cv);
    const int *fi = reinterpret_cast<const int *>(ci);
#pragma unroll
    for (int j = 0; j < kTopK; ++j)
      if (!cand_insert(L, I, fv[j], fi[j])) break;
  }
  for (int rnd = 0; rnd < kTopK; ++rnd) {
    float bv = L[0];
    int bi = I[0];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (cand_better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (I[0] == bi && L[0] == bv) {
#pragma unroll
      for (int j = 0; j < kTopK - 1; ++j) {
        L[j] = L[j + 1];
        I[j] = I[j + 1];
      }
      L[kTopK - 1] = -INFINITY;
      I[kTopK - 1] = 0x7fffffff;
    }
    if (lane == 0) {
      wv[warp][rnd] = bv;
      wi[warp][rnd] = bi;
    }
  }
  __syncthreads();
  if (warp != 0) return;
  int ptr = 0;  // lane w < 8 walks warp w's list
  const size_t o = (static_cast<size_t>(row) * gridDim.x + slice) * kTopK;
  for (int rnd = 0; rnd < kTopK; ++rnd) {
    float bv = (lane < 8 && ptr < kTopK) ? wv[lane][ptr] : -INFINITY;
    int bi = (lane < 8 && ptr < kTopK) ? wi[lane][ptr] : 0x7fffffff;
    const float mv = bv;
    const int mi = bi;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (cand_better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane < 8 && mi == bi && mv == bv) ++ptr;
    if (lane == 0) {
      part_val[o + rnd] = bv;
      part_idx[o + rnd] = bi;
    }
  }
}

// Top-k merge, stage 2: one warp per row merges the row's slice lists (lane s walks list
// s) and writes the k best.
__global__ void __launch_bounds__(32) topk_final_kernel(const float *part_val,
                                                        const int32_t *part_idx, int slices,
                                                        int k, int32_t *tok_out,
                                                        float *score_out) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x, lane = threadIdx.x;
  const size_t base = (static_cast<size_t>(row) * slices + lane) * kTopK;
  int ptr = 0;
  for (int rnd = 0; rnd < k; ++rnd) {
    const bool has = lane < slices && ptr < kTopK;
    float bv = has ? part_val[base + ptr] : -INFINITY;
    int bi = has ? part_idx[base + ptr] : 0x7fffffff;
    const float mv = bv;
    const int mi = bi;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (cand_better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (has && mi == bi && mv == bv) ++ptr;
    if (lane == 0) {
      tok_out[static_cast<size_t>(row) * k + rnd] = bi;
      if (score_out) score_out[static_cast<size_t>(row) * k + rnd] = bv;
    }
  }
}

// fp32 rows -> bf16 hi rows [0, rows) and lo rows [lo_row, lo_row + rows).
// fp32 -> fp16 (the operand type of the head's products when its packed copy is fp16).
__global__ void rows_f16_kernel(const float *src, size_t n, __half *dst, ZeroSpan z) {
  pdl_wait();
  pdl_trigger();
  zero_span(z);
  for (size_t t = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; t < n;
       t += static_cast<size_t>(gridDim.x) * blockDim.x) {
    flag_f16_range(f16_out_of_range(src[t]));
    dst[t] = __float2half_rn(src[t]);
  }
}

__global__ void split_rows_kernel(const float *src, size_t n, __nv_bfloat16 *dst, size_t lo_off,
                                  ZeroSpan z) {
  pdl_wait();
  pdl_trigger();
  zero_span(z);
  for (size_t t = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; t < n;
       t += static_cast<size_t>(gridDim.x) * blockDim.x)
    store_split(dst, t, lo_off, src[t]);
}

__global__ void zero_kernel(ZeroSpan z) {
  pdl_wait();
  pdl_trigger();
  zero_span(z);
}

__global__ void copy_f32_kernel(const float *src, float *dst, size_t n) {
  pdl_wait();
  pdl_trigger();
  for (size_t t = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; t < n;
       t += static_cast<size_t>(gridDim.x) * blockDim.x)
    dst[t] = src[t];
}

// ------------------------------------------------------------------ last-write refinement
// "DSpine 完全拆解", section on predecessor-conditioned decoding and the transition cache.

// The last layer's state the refinement redoes its injection from: the pre-injection
// residual u [T][H], the receiver RMS r [T] and the receiver gate term G c [T][Mc]
// (columns 0..Mc of the gate-map GEMM output pre [T][3 Mc]).
__global__ void tail_export_kernel(const float *x, const float *r, const float *pre, int T, int H,
                                   int Mc, float *out) {
  pdl_wait();
  pdl_trigger();
  const size_t nx = static_cast<size_t>(T) * H, ng = static_cast<size_t>(T) * Mc;
  for (size_t t = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; t < nx + T + ng;
       t += static_cast<size_t>(gridDim.x) * blockDim.x) {
    if (t < nx) {
      out[t] = x[t];
    } else if (t < nx + T) {
      out[t] = r[t - nx];
    } else {
      const size_t g = t - nx - T;
      out[t] = pre[(g / Mc) * 3 * Mc + g % Mc];
    }
  }
}

// Pair n = ((b * (K - 1) + (i - 2)) * kc + p) takes predecessor candidate p of block row
// i - 1: its codebook row, for the predecessor-gate and value maps.
template <typename T, typename O>
__global__ void tail_gather_kernel(const T *codebook, int V, int Rc, const int32_t *cand, int K,
                                   int kc, int n_pairs, O *out) {
  pdl_wait();
  pdl_trigger();
  const int n = blockIdx.x;
  if (n >= n_pairs) return;
  const int p = n % kc, bi = n / kc, b = bi / (K - 1), i = bi % (K - 1) + 2;
  int s = cand[(static_cast<size_t>(b) * K + (i - 2)) * kc + p];
  if (s < 0 || s >= V) {
    if (threadIdx.x == 0) atomicOr(&g_error_word, DEVERR_BAD_INDEX);
    s = 0;
  }
  const T *src = codebook + static_cast<size_t>(s) * Rc;
  for (int k = threadIdx.x; k < Rc; k += blockDim.x)
    out[static_cast<size_t>(n) * Rc + k] = from_f<O>(to_f<T>(src[k]));
}

// m = sigmoid(G c_i + sqrt(Rc) G_p C_s + b) * (sqrt(Rc) A C_s) for pair n (row i of request
// b); pre2 [n][2 Mc] = [G_p C_s, A C_s]; written as the write GEMM's operand (an fp16 row,
// or a bf16 hi+lo pair).
template <typename T, typename O>
__global__ void tail_message_kernel(const float *pre2, const float *gc, const T *bias, int K, int W,
                                    int kc, int Mc, float scale, O *m_out, size_t lo_off) {
  pdl_wait();
  pdl_trigger();
  const int n = blockIdx.x;
  const int bi = n / kc, b = bi / (K - 1), i = bi % (K - 1) + 2;
  const float *g_recv = gc + (static_cast<size_t>(b) * W + i) * Mc;
  const float *pp = pre2 + static_cast<size_t>(n) * 2 * Mc;
  for (int f = threadIdx.x; f < Mc; f += blockDim.x) {
    const float z = g_recv[f] + scale * pp[f] + (bias ? to_f<T>(bias[f]) : 0.f);
    const float g = 1.f / (1.f + expf(-z));
    store_split(m_out + static_cast<size_t>(n) * Mc, f, lo_off, g * scale * pp[Mc + f]);
  }
}

// Eight consecutive elements as fp32 (one 16-byte load for bf16, two for fp32).
template <typename T> __device__ __forceinline__ void load8(const T *p, float (&o)[8]);
template <> __device__ __forceinline__ void load8<float>(const float *p, float (&o)[8]) {
  const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}
template <> __device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16 *p, float (&o)[8]) {
  const uint4 u = *reinterpret_cast<const uint4 *>(p);
  const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 f = __bfloat1622float2(h[q]);
    o[2 * q] = f.x;
    o[2 * q + 1] = f.y;
  }
}

// One CTA per predecessor pair n (request b, block row i >= 2, candidate p of row i-1):
// the refined state x' = u_i + r_i delta_n goes through the final norm and is scored
// against the head rows of row i's kc candidates.  Two passes over H in 8-element vectors
// (the mean square, then the dot products); the pairs of one row share the candidate head
// rows through L2.  Requires H % 8 == 0.
template <typename T>
__global__ void __launch_bounds__(256) tail_scores_kernel(const float *u, const float *r,
                                                          const float *delta, const T *embed,
                                                          const T *gain, const int32_t *cand,
                                                          int K, int W, int kc, int H, int V,
                                                          float eps, float *table) {
  __shared__ float part[8][kTopK + 1];
  __shared__ int cid[kTopK];
  __shared__ float s_inv;
  pdl_wait();
  pdl_trigger();
  const int n = blockIdx.x, bi = n / kc, b = bi / (K - 1), i = bi % (K - 1) + 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t t = static_cast<size_t>(b) * W + i;  // the block row
  const float *ut = u + t * H;
  const float *dn = delta + static_cast<size_t>(n) * H;
  const float rt = r[t];
  if (threadIdx.x < kc) {
    int c = cand[(static_cast<size_t>(b) * K + (i - 1)) * kc + threadIdx.x];
    if (c < 0 || c >= V) {
      atomicOr(&g_error_word, DEVERR_BAD_INDEX);
      c = 0;
    }
    cid[threadIdx.x] = c;
  }
  float ss = 0.f;
  for (int d = threadIdx.x * 8; d < H; d += blockDim.x * 8) {
    float uu[8], dd[8];
    load8<float>(ut + d, uu);
    load8<float>(dn + d, dd);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float x = uu[q] + rt * dd[q];
      ss += x * x;
    }
  }
  ss = warp_sum(ss);
  if (lane == 0) part[warp][0] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int w = 0; w < 8; ++w) tot += part[w][0];
    s_inv = rsqrtf(tot / static_cast<float>(H) + eps);
  }
  __syncthreads();
  const float inv = s_inv;
  float acc[kTopK];
#pragma unroll
  for (int j = 0; j < kTopK; ++j) acc[j] = 0.f;
  for (int d = threadIdx.x * 8; d < H; d += blockDim.x * 8) {
    float uu[8], dd[8], gg[8], h[8];
    load8<float>(ut + d, uu);
    load8<float>(dn + d, dd);
    load8<T>(gain + d, gg);
#pragma unroll
    for (int q = 0; q < 8; ++q) h[q] = gg[q] * (uu[q] + rt * dd[q]) * inv;
#pragma unroll
    for (int j = 0; j < kTopK; ++j) {
      if (j < kc) {
        float e[8];
        load8<T>(embed + static_cast<size_t>(cid[j]) * H + d, e);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[j] += h[q] * e[q];
      }
    }
  }
  __syncthreads();  // part[] is reused
#pragma unroll
  for (int j = 0; j < kTopK; ++j) {
    const float v = warp_sum(acc[j]);
    if (lane == 0) part[warp][j] = v;
  }
  __syncthreads();
  if (threadIdx.x < kc) {
    float tot = 0.f;
    for (int w = 0; w < 8; ++w) tot += part[w][threadIdx.x];
    table[static_cast<size_t>(n) * kc + threadIdx.x] = tot;
  }
}

// Greedy walk of request b (one warp, the request's tables staged in shared memory):
// row 1 takes the lowest-rank best of its own scores, row i >= 2 the lowest-rank best of
// the table row of row i - 1's choice.
__global__ void __launch_bounds__(32) tail_walk_kernel(const float *table, const float *cand_score,
                                                       const int32_t *cand, int K, int kc,
                                                       int32_t *token_out, int32_t *pick_out) {
  extern __shared__ float tb[];  // [(K - 1) * kc * kc]
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, lane = threadIdx.x;
  const size_t tsz = static_cast<size_t>(K - 1) * kc * kc;
  for (size_t q = lane; q < tsz; q += 32) tb[q] = table[b * tsz + q];
  __syncwarp();
  auto best = [&](float v) {  // lowest lane among the maxima of lanes < kc
    float bv = lane < kc ? v : -INFINITY;
    int bl = lane < kc ? lane : 0x7fffffff;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int ol = __shfl_xor_sync(0xffffffffu, bl, off);
      if (ov > bv || (ov == bv && ol < bl)) {
        bv = ov;
        bl = ol;
      }
    }
    return bl;
  };
  int j = best(lane < kc ? cand_score[static_cast<size_t>(b) * K * kc + lane] : 0.f);
  if (lane == 0) {
    token_out[static_cast<size_t>(b) * K] = cand[static_cast<size_t>(b) * K * kc + j];
    if (pick_out) pick_out[static_cast<size_t>(b) * K] = j;
  }
  for (int i = 2; i <= K; ++i) {
    const float v = lane < kc ? tb[(static_cast<size_t>(i - 2) * kc + j) * kc + lane] : 0.f;
    j = best(v);
    if (lane == 0) {
      const size_t row = static_cast<size_t>(b) * K + (i - 1);
      token_out[row] = cand[row * kc + j];
      if (pick_out) pick_out[row] = j;
    }
  }
}

// Self-test of the failure path: one thread waits, bounded, for a counter that only the
// caller sets, with the same wait the split-tile reductions and attention splits use.
__global__ void wait_selftest_kernel(const unsigned *flag, unsigned long long limit_ns) {
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) wait_count(flag, 1u, limit_ns);
}

// ------------------------------------------------------------------ launchers
static std::string err(const char *what, cudaError_t e) {
  return e == cudaSuccess ? std::string() : std::string(what) + ": " + cudaGetErrorString(e);
}

std::string launch_round_prep(int dtype, const void *embed, int H, int V, const int32_t *anchors,
                              const int64_t *frontier, int B, int W, int mask_id, float *x,
                              float2 *rope, int half, const RopeFreq &freq, const int64_t *pend_pos,
                              int n_pend, ZeroSpan z, cudaStream_t s) {
  cudaError_t e;
  const int T = B * W;
  if (dtype == 0)
    e = launch_pdl(round_prep_kernel<__nv_bfloat16>, dim3(T + n_pend), dim3(256), 0, s,
                   static_cast<const __nv_bfloat16 *>(embed), H, V, anchors, frontier, W, T, mask_id,
                   x, rope, half, freq, pend_pos, z);
  else
    e = launch_pdl(round_prep_kernel<float>, dim3(T + n_pend), dim3(256), 0, s,
                   static_cast<const float *>(embed), H, V, anchors, frontier, W, T, mask_id, x,
                   rope, half, freq, pend_pos, z);
  return err("round prep", e);
}

std::string launch_rope_table(const int64_t *pos, int n, float2 *rope, int half,
                              const RopeFreq &freq, ZeroSpan z, cudaStream_t s) {
  const int total = n * half;
  const int blocks = (total + 255) / 256;
  return err("rope table", launch_pdl(rope_table_kernel, dim3(blocks < 1024 ? blocks : 1024),
                                      dim3(256), 0, s, pos, n, rope, half, freq, z));
}

std::string launch_zero(ZeroSpan z, cudaStream_t s) {
  const size_t blocks = (z.n + 255) / 256;
  return err("zero", launch_pdl(zero_kernel, dim3(blocks < 64 ? (blocks > 0 ? blocks : 1) : 64),
                                dim3(256), 0, s, z));
}

std::string launch_rownorm(int dtype, float *x, int rows, int H, const void *gain, float eps,
                           int mode, void *out, float *r_out, float *f32_out, float *head_out, int W,
                           size_t lo_off, cudaStream_t s, const ConvFinish &cf, bool out_f16) {
  cudaError_t e;
  if (dtype == 0 && out_f16)
    e = launch_pdl(rownorm_kernel<__nv_bfloat16, __half>, dim3(rows), dim3(256), 0, s, x, H,
                   static_cast<const __nv_bfloat16 *>(gain), eps, mode, static_cast<__half *>(out),
                   r_out, f32_out, head_out, W, lo_off, cf);
  else if (dtype == 0)
    e = launch_pdl(rownorm_kernel<__nv_bfloat16, __nv_bfloat16>, dim3(rows), dim3(256), 0, s, x,
                   H, static_cast<const __nv_bfloat16 *>(gain), eps, mode,
                   static_cast<__nv_bfloat16 *>(out), r_out, f32_out, head_out, W, lo_off, cf);
  else
    e = launch_pdl(rownorm_kernel<float, float>, dim3(rows), dim3(256), 0, s, x, H,
                   static_cast<const float *>(gain), eps, mode, static_cast<float *>(out), r_out,
                   f32_out, head_out, W, lo_off, cf);
  return err("rownorm", e);
}

std::string launch_conv_prepare(int dtype, const float *X, const float *delta, const void *base,
                                int rows, int H, int gw, int W, void *out, size_t lo_off,
                                cudaStream_t s, bool out_f16) {
  cudaError_t e;
  if (dtype == 0 && out_f16)
    e = launch_pdl(conv_prepare_kernel<__nv_bfloat16, __half>, dim3(rows), dim3(256), 0, s, X,
                   delta, static_cast<const __nv_bfloat16 *>(base), H, gw, W,
                   static_cast<__half *>(out), lo_off);
  else if (dtype == 0)
    e = launch_pdl(conv_prepare_kernel<__nv_bfloat16, __nv_bfloat16>, dim3(rows), dim3(256), 0, s,
                   X, delta, static_cast<const __nv_bfloat16 *>(base), H, gw, W,
                   static_cast<__nv_bfloat16 *>(out), lo_off);
  else
    e = launch_pdl(conv_prepare_kernel<float, float>, dim3(rows), dim3(256), 0, s, X, delta,
                   static_cast<const float *>(base), H, gw, W, static_cast<float *>(out), lo_off);
  return err("conv prepare", e);
}

std::string launch_rows_f16(const float *src, size_t n, void *dst, ZeroSpan z, cudaStream_t s) {
  const size_t blocks = (n + 255) / 256;
  return err("fp16 rows", launch_pdl(rows_f16_kernel, dim3(blocks < 2048 ? blocks : 2048),
                                     dim3(256), 0, s, src, n, static_cast<__half *>(dst), z));
}

std::string launch_split_rows(const float *src, size_t n, void *dst, size_t lo_off, ZeroSpan z,
                              cudaStream_t s) {
  const size_t blocks = (n + 255) / 256;
  return err("split rows", launch_pdl(split_rows_kernel, dim3(blocks < 2048 ? blocks : 2048),
                                      dim3(256), 0, s, src, n, static_cast<__nv_bfloat16 *>(dst),
                                      lo_off, z));
}

std::string launch_head_post(int dtype, const HeadPostArgs &a, cudaStream_t s) {
  const long long warps = static_cast<long long>(a.rows) * a.total_heads;
  const dim3 grid(static_cast<unsigned>((warps + 7) / 8));
  cudaError_t e;
  if (a.D == 128)
    e = dtype == 0 ? launch_pdl(head_post_kernel<__nv_bfloat16, 4>, grid, dim3(256), 0, s, a)
                   : launch_pdl(head_post_kernel<float, 4>, grid, dim3(256), 0, s, a);
  else
    e = dtype == 0 ? launch_pdl(head_post_kernel<__nv_bfloat16, 2>, grid, dim3(256), 0, s, a)
                   : launch_pdl(head_post_kernel<float, 2>, grid, dim3(256), 0, s, a);
  return err("head post", e);
}

std::string launch_code(int dtype, const float *z, int rows, int Rc, const void *codebook,
                        const int32_t *anchors, int V, int W, float eps, void *c_out,
                        size_t lo_off, cudaStream_t s, bool out_f16) {
  cudaError_t e;
  if (dtype == 0 && out_f16)
    e = launch_pdl(code_kernel<__nv_bfloat16, __half>, dim3(rows), dim3(256), 0, s, z, Rc,
                   static_cast<const __nv_bfloat16 *>(codebook), anchors, V, W, eps,
                   static_cast<__half *>(c_out), static_cast<size_t>(0));
  else if (dtype == 0)
    e = launch_pdl(code_kernel<__nv_bfloat16, __nv_bfloat16>, dim3(rows), dim3(256), 0, s, z, Rc,
                   static_cast<const __nv_bfloat16 *>(codebook), anchors, V, W, eps,
                   static_cast<__nv_bfloat16 *>(c_out), lo_off);
  else
    e = launch_pdl(code_kernel<float, float>, dim3(rows), dim3(256), 0, s, z, Rc,
                   static_cast<const float *>(codebook), anchors, V, W, eps,
                   static_cast<float *>(c_out), lo_off);
  return err("code", e);
}

std::string launch_message(int dtype, const float *pre, int rows, int Mc, const void *bias, int W,
                           void *m_out, size_t lo_off, cudaStream_t s, bool out_f16) {
  cudaError_t e;
  if (dtype == 0 && out_f16)
    e = launch_pdl(message_kernel<__nv_bfloat16, __half>, dim3(rows), dim3(256), 0, s, pre, Mc,
                   static_cast<const __nv_bfloat16 *>(bias), W, static_cast<__half *>(m_out),
                   static_cast<size_t>(0));
  else if (dtype == 0)
    e = launch_pdl(message_kernel<__nv_bfloat16, __nv_bfloat16>, dim3(rows), dim3(256), 0, s, pre,
                   Mc, static_cast<const __nv_bfloat16 *>(bias), W,
                   static_cast<__nv_bfloat16 *>(m_out), lo_off);
  else
    e = launch_pdl(message_kernel<float, float>, dim3(rows), dim3(256), 0, s, pre, Mc,
                   static_cast<const float *>(bias), W, static_cast<float *>(m_out), lo_off);
  return err("message", e);
}

std::string launch_argmax_reduce(const float *val, const int32_t *idx, int m_tiles, int rows,
                                 int32_t *tok_out, float *max_out, cudaStream_t s) {
  return err("argmax reduce", launch_pdl(argmax_reduce_kernel, dim3(rows), dim3(256), 0, s, val,
                                         idx, m_tiles, rows, tok_out, max_out));
}

int topk_slices(int m_tiles) { return (m_tiles + kTopKTilesPerSlice - 1) / kTopKTilesPerSlice; }

std::string launch_topk_reduce(const float *val, const int32_t *idx, int m_tiles, int rows, int k,
                               float *part_val, int32_t *part_idx, int32_t *tok_out,
                               float *score_out, cudaStream_t s) {
  const int slices = topk_slices(m_tiles);
  if (slices > 32) return "top-k reduce: vocabulary too large";
  cudaError_t e = launch_pdl(topk_slice_kernel, dim3(slices, rows), dim3(256), 0, s, val, idx,
                             m_tiles, rows, kTopKTilesPerSlice, part_val, part_idx);
  if (e == cudaSuccess)
    e = launch_pdl(topk_final_kernel, dim3(rows), dim3(32), 0, s, part_val, part_idx, slices, k,
                   tok_out, score_out);
  return err("top-k reduce", e);
}

std::string launch_copy_f32(const float *src, float *dst, size_t n, cudaStream_t s) {
  const size_t blocks = (n + 255) / 256;
  return err("copy", launch_pdl(copy_f32_kernel, dim3(blocks < 1024 ? blocks : 1024), dim3(256), 0,
                                s, src, dst, n));
}

}  // namespace bd

namespace bd {

std::string launch_tail_export(const float *x, const float *r, const float *pre, int T, int H,
                               int Mc, float *out, cudaStream_t s) {
  const size_t n = static_cast<size_t>(T) * (H + 1 + Mc);
  const size_t blocks = (n + 255) / 256;
  return err("tail export", launch_pdl(tail_export_kernel, dim3(blocks < 1024 ? blocks : 1024),
                                       dim3(256), 0, s, x, r, pre, T, H, Mc, out));
}

std::string launch_tail_gather(int dtype, const void *codebook, int V, int Rc, const int32_t *cand,
                               int K, int kc, int n_pairs, void *out, cudaStream_t s, bool out_f16) {
  cudaError_t e;
  if (dtype == 0 && out_f16)
    e = launch_pdl(tail_gather_kernel<__nv_bfloat16, __half>, dim3(n_pairs), dim3(128), 0, s,
                   static_cast<const __nv_bfloat16 *>(codebook), V, Rc, cand, K, kc, n_pairs,
                   static_cast<__half *>(out));
  else if (dtype == 0)
    e = launch_pdl(tail_gather_kernel<__nv_bfloat16, __nv_bfloat16>, dim3(n_pairs), dim3(128), 0, s,
                   static_cast<const __nv_bfloat16 *>(codebook), V, Rc, cand, K, kc, n_pairs,
                   static_cast<__nv_bfloat16 *>(out));
  else
    e = launch_pdl(tail_gather_kernel<float, float>, dim3(n_pairs), dim3(128), 0, s,
                   static_cast<const float *>(codebook), V, Rc, cand, K, kc, n_pairs,
                   static_cast<float *>(out));
  return err("tail gather", e);
}

std::string launch_tail_message(int dtype, const float *pre2, const float *gc, const void *bias, int K,
                                int W, int kc, int Mc, float scale, int n_pairs, void *m_out,
                                size_t lo_off, cudaStream_t s, bool out_f16) {
  cudaError_t e;
  if (dtype == 0 && out_f16)
    e = launch_pdl(tail_message_kernel<__nv_bfloat16, __half>, dim3(n_pairs), dim3(128), 0, s, pre2,
                   gc, static_cast<const __nv_bfloat16 *>(bias), K, W, kc, Mc, scale,
                   static_cast<__half *>(m_out), static_cast<size_t>(0));
  else if (dtype == 0)
    e = launch_pdl(tail_message_kernel<__nv_bfloat16, __nv_bfloat16>, dim3(n_pairs), dim3(128), 0, s,
                   pre2, gc, static_cast<const __nv_bfloat16 *>(bias), K, W, kc, Mc, scale,
                   static_cast<__nv_bfloat16 *>(m_out), lo_off);
  else
    e = launch_pdl(tail_message_kernel<float, float>, dim3(n_pairs), dim3(128), 0, s, pre2, gc,
                   static_cast<const float *>(bias), K, W, kc, Mc, scale,
                   static_cast<float *>(m_out), lo_off);
  return err("tail message", e);
}

std::string launch_tail_scores(int dtype, const float *u, const float *r, const float *delta,
                               const void *embed, const void *gain, const int32_t *cand, int B, int K,
                               int W, int kc, int H, int V, float eps, float *table, cudaStream_t s) {
  cudaError_t e;
  const dim3 grid(B * (K - 1) * kc);  // one CTA per predecessor pair
  if (H % 8 != 0) return "tail scores: hidden size must be a multiple of 8";
  if (dtype == 0)
    e = launch_pdl(tail_scores_kernel<__nv_bfloat16>, grid, dim3(256), 0, s, u, r, delta,
                   static_cast<const __nv_bfloat16 *>(embed),
                   static_cast<const __nv_bfloat16 *>(gain), cand, K, W, kc, H, V, eps, table);
  else
    e = launch_pdl(tail_scores_kernel<float>, grid, dim3(256), 0, s, u, r, delta,
                   static_cast<const float *>(embed), static_cast<const float *>(gain), cand, K, W,
                   kc, H, V, eps, table);
  return err("tail scores", e);
}

std::string launch_tail_walk(const float *table, const float *cand_score, const int32_t *cand, int B,
                             int K, int kc, int32_t *token_out, int32_t *pick_out, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(K - 1) * kc * kc * sizeof(float);
  return err("tail walk", launch_pdl(tail_walk_kernel, dim3(B), dim3(32), smem, s, table, cand_score,
                                     cand, K, kc, token_out, pick_out));
}

std::string launch_wait_selftest(const unsigned *flag, unsigned long long limit_ns, cudaStream_t s) {
  return err("wait self-test", launch_pdl(wait_selftest_kernel, dim3(1), dim3(32), 0, s, flag, limit_ns));
}

}  // namespace bd
