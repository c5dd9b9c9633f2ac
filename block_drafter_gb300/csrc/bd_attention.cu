// Block attention of the drafter: the W block rows of a request attend over the
// request's ring context plus the block's own keys ([DFlash-notes] per-layer equations
// and local-window rule; [BlockCausal] for the optional block-causal mask):
//
//   a = softmax(q K^T / sqrt(D) + mask) V,  K = [K_ctx; k_block], V = [V_ctx; v_block]
//
// A context key at position p is visible from block row i (position F+i) iff
// (F+i) - p < S for a local layer; every populated position for a full layer.  Block
// key j is visible iff |j - i| < S (local) and, block-causal, j <= i.
//
// bf16 path: one CTA per (key split, KV head, request).  All G = Hq/Hkv query heads of
// the KV head and all W rows (G*W <= 64 query rows) share each K/V tile, so the
// windowed context is streamed once per KV head.  QK^T and PV run on mma.sync bf16
// tensor-core instructions with an online (max-subtracted, base-2) softmax; each split
// writes an unnormalised partial (O, m, l) and a combine kernel merges the splits.
#include "bd_device.cuh"
#include "bd_internal.h"
#include "bd_kernels.h"

#include <climits>

namespace bd {

BD_DEFINE_ERROR_TAKER(take_error_word_att)

constexpr int kAttRows = 64;     // query rows per CTA (4 warps x 16)
constexpr int kAttKeys = 64;     // keys per pipeline block
constexpr int kAttPad = 8;       // bf16 padding per smem row (bank-conflict-free ldmatrix)

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                          uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
      "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma16816_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
      "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// 8 bf16 values (16 bytes of shared memory) rewritten in place as fp16, saturating at
// +-65504 (exact for every bf16 value of magnitude 2^-14 .. 65504).
__device__ __forceinline__ void bf16x8_to_f16_inplace(__nv_bfloat16 *p) {
  uint4 v = *reinterpret_cast<const uint4 *>(p);
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
    f.x = fminf(fmaxf(f.x, -65504.f), 65504.f);
    f.y = fminf(fmaxf(f.y, -65504.f), 65504.f);
    const __half2 h = __floats2half2_rn(f.x, f.y);
    w[i] = *reinterpret_cast<const uint32_t *>(&h);
  }
  *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ uint32_t pack_f16(float x0, float x1) {
  const __half2 h = __floats2half2_rn(x0, x1);
  return *reinterpret_cast<const uint32_t *>(&h);
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

struct AttGeom {
  long long F;
  int p_lo, n_ctx, k_begin, k_end;
};

// Context keys [p_lo, F) of request b (the window's oldest visible position, clipped to
// the ring's live interval) are split into chunks of whole 64-key blocks: one per split,
// or one per split but the last when that split only takes the block's own keys.
__device__ __forceinline__ AttGeom att_geom(const AttArgs &a, int b, int split) {
  AttGeom g;
  g.F = a.frontier[b];
  long long lo = a.window > 0 ? g.F - a.window + 1 : 0;
  if (g.F - a.cap > lo) lo = g.F - a.cap;  // the ring holds [F - cap, F)
  if (lo < 0) lo = 0;
  g.p_lo = static_cast<int>(lo);
  g.n_ctx = g.F > lo ? static_cast<int>(g.F - lo) : 0;
  const int cs = a.block_split ? a.n_splits - 1 : a.n_splits;  // splits with context keys
  int chunk = (g.n_ctx + cs - 1) / cs;
  chunk = (chunk + kAttKeys - 1) / kAttKeys * kAttKeys;
  g.k_begin = min(g.n_ctx, split * chunk);
  g.k_end = min(g.n_ctx, g.k_begin + chunk);
  return g;
}

// Is context key k (0-based from p_lo) visible from block row i?
__device__ __forceinline__ bool ctx_visible(const AttArgs &a, const AttGeom &g, int i, int k) {
  if (k >= g.k_end) return false;
  const long long p = g.p_lo + k;
  return a.window <= 0 || (g.F + i) - p < a.window;
}
// Is block key j visible from block row i?
__device__ __forceinline__ bool blk_visible(const AttArgs &a, int i, int j) {
  if (j >= a.W) return false;
  if (a.window > 0 && abs(j - i) >= a.window) return false;
  return !a.causal || j <= i;
}

// hi/lo split of a probability pair for the bf16 A operand of P.V
__device__ __forceinline__ void split_pack(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t *>(&h);
  lo = *reinterpret_cast<const uint32_t *>(&l);
}

// Online-softmax update of one warp's 16 rows for a tile of NT*8 keys (scores already
// scaled to log2 units and masked with -inf); returns the probabilities in s.
template <int NT>
__device__ __forceinline__ void softmax_update(float (&s)[NT][4], float (&m_run)[2],
                                               float (&l_run)[2], float (&alpha)[2]) {
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) mx[e >> 1] = fmaxf(mx[e >> 1], s[nt][e]);
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 1));
    mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 2));
    const float m_new = fmaxf(m_run[hr], mx[hr]);
    alpha[hr] = (m_new == -INFINITY) ? 1.f : exp2f(m_run[hr] - m_new);
    m_run[hr] = m_new;
  }
  float ls[2] = {0.f, 0.f};
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int hr = e >> 1;
      const float pv = (s[nt][e] == -INFINITY) ? 0.f : exp2f(s[nt][e] - m_run[hr]);
      s[nt][e] = pv;
      ls[hr] += pv;
    }
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    ls[hr] += __shfl_xor_sync(0xffffffffu, ls[hr], 1);
    ls[hr] += __shfl_xor_sync(0xffffffffu, ls[hr], 2);
    l_run[hr] = l_run[hr] * alpha[hr] + ls[hr];
  }
}

// Merge the splits of query rows r0 .. r1-1 of (request b, KV head h):
//   out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
// The four warps take (row, part) tasks: with fewer than three rows each row's splits are
// shared by 4 / rows warps, whose sums meet in shared memory.  Lanes own D/32 consecutive
// output dims; split weights are computed by lanes and broadcast, and the partial tiles are
// loaded eight splits at a time before they are used (the loads are independent and their
// L2 latency, not bandwidth, bounds the merge).  The partials were written by other CTAs of
// the launch: read through L2.  Called by all threads of the CTA.
// Few splits (S <= SMAX): each warp merges rows r0 + warp, r0 + warp + 4, ... RB at a time,
// with every load of those rows (the splits' (m, l) and partial rows) issued before any
// arithmetic, so they cost one round trip to L2.  Splits are added in index order.
constexpr int kFewSplits = 8;
template <typename T, int D, int SMAX, int RB>
__device__ __forceinline__ void combine_rows_few(const AttArgs &a, int b, int h, int r0, int r1,
                                                 int warp, int lane) {
  constexpr int PER = D / 32;
  const int G = a.n_q_heads / a.n_kv_heads, S = a.n_splits;
  const size_t bh = static_cast<size_t>(b) * a.n_kv_heads + h;
  const float *po = a.part_o + bh * S * kAttRows * D;
  const float2 *pml = a.part_ml + bh * S * kAttRows;
  for (int base = r0 + warp; base < r1; base += 4 * RB) {
    float2 ml[RB][SMAX];
    float v[RB][SMAX][PER];
#pragma unroll
    for (int i = 0; i < RB; ++i) {
      const int rr = base + 4 * i;
#pragma unroll
      for (int sp = 0; sp < SMAX; ++sp) {
        const bool ok = rr < r1 && sp < S;
        ml[i][sp] = ok ? __ldcg(pml + sp * kAttRows + rr) : make_float2(-INFINITY, 0.f);
        const float *os = po + (static_cast<size_t>(ok ? sp : 0) * kAttRows + (ok ? rr : 0)) * D + lane * PER;
        if (PER == 4) {
          const float4 o = ok ? __ldcg(reinterpret_cast<const float4 *>(os)) : make_float4(0.f, 0.f, 0.f, 0.f);
          v[i][sp][0] = o.x;
          v[i][sp][1 % PER] = o.y;
          v[i][sp][2 % PER] = o.z;
          v[i][sp][3 % PER] = o.w;
        } else {
          const float2 o = ok ? __ldcg(reinterpret_cast<const float2 *>(os)) : make_float2(0.f, 0.f);
          v[i][sp][0] = o.x;
          v[i][sp][1 % PER] = o.y;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < RB; ++i) {
      const int rr = base + 4 * i;
      if (rr >= r1) break;
      float M = -INFINITY;
#pragma unroll
      for (int sp = 0; sp < SMAX; ++sp)
        if (ml[i][sp].y > 0.f) M = fmaxf(M, ml[i][sp].x);
      float L = 0.f, acc[PER];
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] = 0.f;
#pragma unroll
      for (int sp = 0; sp < SMAX; ++sp)
        if (ml[i][sp].y > 0.f) {
          const float wgt = exp2f(ml[i][sp].x - M);
          L += wgt * ml[i][sp].y;
#pragma unroll
          for (int e = 0; e < PER; ++e) acc[e] += wgt * v[i][sp][e];
        }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      const int gh = rr / a.W, qi = rr % a.W;
      T *out = static_cast<T *>(a.out) +
               (static_cast<size_t>(b) * a.W + qi) * a.n_q_heads * D + (h * G + gh) * D + lane * PER;
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        const float y = acc[e] * inv;
        const T hi = from_f<T>(y);
        out[e] = hi;
        if (a.out_lo) out[a.out_lo + e] = from_f<T>(y - to_f<T>(hi));
      }
    }
  }
}

template <typename T, int D>
__device__ __forceinline__ void combine_rows(const AttArgs &a, int b, int h, int r0, int r1,
                                             int warp, int lane, float (*red)[D + 4]) {
  const int G = a.n_q_heads / a.n_kv_heads;
  const size_t bh = static_cast<size_t>(b) * a.n_kv_heads + h;
  constexpr int PER = D / 32;
  constexpr int kBatch = 8;
  const float *po = a.part_o + bh * a.n_splits * kAttRows * D;
  const float2 *pml = a.part_ml + bh * a.n_splits * kAttRows;
  const int nrows = r1 - r0;
  const int P = nrows >= 3 ? 1 : 4 / max(nrows, 1);  // warps per row
  const int S = a.n_splits;
  for (int t0 = 0; t0 < nrows * P; t0 += 4) {
    const int t = t0 + warp;
    const bool active = t < nrows * P;
    const int rr = r0 + (active ? t / P : 0), part = t % P;
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    float L = 0.f;
    if (active) {
      float M = -INFINITY;
      for (int s = lane; s < S; s += 32) {
        const float2 ml = __ldcg(pml + s * kAttRows + rr);
        if (ml.y > 0.f) M = fmaxf(M, ml.x);
      }
      M = warp_max(M);
      const int s_begin = part * S / P, s_end = (part + 1) * S / P;
      for (int s0 = s_begin; s0 < s_end; s0 += 32) {
        const int s = s0 + lane;
        float wgt = 0.f;
        if (s < s_end) {
          const float2 ml = __ldcg(pml + s * kAttRows + rr);
          if (ml.y > 0.f) {
            wgt = exp2f(ml.x - M);
            L += wgt * ml.y;
          }
        }
        const int cnt = min(32, s_end - s0);
        for (int j0 = 0; j0 < cnt; j0 += kBatch) {
          float v[kBatch][PER];
#pragma unroll
          for (int u = 0; u < kBatch; ++u) {
            const float *os = po + (static_cast<size_t>(s0 + j0 + u) * kAttRows + rr) * D + lane * PER;
            if (j0 + u < cnt) {
              if (PER == 4) {
                const float4 o = __ldcg(reinterpret_cast<const float4 *>(os));
                v[u][0] = o.x;
                v[u][1] = o.y;
                v[u][2] = o.z;
                v[u][3] = o.w;
              } else {
                const float2 o = __ldcg(reinterpret_cast<const float2 *>(os));
                v[u][0] = o.x;
                v[u][1] = o.y;
              }
            }
          }
#pragma unroll
          for (int u = 0; u < kBatch; ++u) {
            const float wj = __shfl_sync(0xffffffffu, wgt, (j0 + u) & 31);
            if (j0 + u < cnt)
#pragma unroll
              for (int e = 0; e < PER; ++e) acc[e] += wj * v[u][e];
          }
        }
      }
      L = warp_sum(L);
    }
    if (P > 1) {  // the parts of a row meet in shared memory
      if (active) {
#pragma unroll
        for (int e = 0; e < PER; ++e) red[warp][lane * PER + e] = acc[e];
        if (lane == 0) red[warp][D] = L;
      }
      __syncthreads();
      if (active && part == 0)
        for (int q = 1; q < P; ++q) {
#pragma unroll
          for (int e = 0; e < PER; ++e) acc[e] += red[warp + q][lane * PER + e];
          L += red[warp + q][D];
        }
    }
    if (active && part == 0) {
      const float inv = L > 0.f ? 1.f / L : 0.f;
      const int gh = rr / a.W, i = rr % a.W;
      T *out = static_cast<T *>(a.out) +
               (static_cast<size_t>(b) * a.W + i) * a.n_q_heads * D + (h * G + gh) * D + lane * PER;
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        const float y = acc[e] * inv;
        const T hi = from_f<T>(y);
        out[e] = hi;
        if (a.out_lo) out[a.out_lo + e] = from_f<T>(y - to_f<T>(hi));
      }
    }
  }
}

// bf16 tensor-core path.  Q and the softmax probabilities P enter the MMAs as hi+lo bf16
// pairs (fp32 accumulate), so their rounding does not reach the output; the ring's K/V
// are exact bf16 data.  The block's own keys/values (produced this round, hi+lo) are
// processed by the last split in a separate 16-key pass.
// F16: Q, P and the block's keys/values are single fp16 operands (11 significant bits) and
// each ring tile is rewritten as fp16 in shared memory once it lands (exact within fp16's
// range): half the MMAs of the hi+lo form.
template <int D, bool F16>
__global__ void __launch_bounds__(128, 2) attention_bf16_kernel(const __grid_constant__ AttArgs a) {
  extern __shared__ uint8_t smem_raw[];
  constexpr int RS = D + kAttPad;  // smem row stride (elements)
  __nv_bfloat16 *sQ = reinterpret_cast<__nv_bfloat16 *>(smem_raw);   // [2][64][RS] hi, lo
  __nv_bfloat16 *sK = sQ + 2 * kAttRows * RS;                          // [2][64][RS]
  __nv_bfloat16 *sV = sK + 2 * kAttKeys * RS;                          // [2][64][RS]

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.n_q_heads / a.n_kv_heads;
  const int R = G * a.W;
  // The frontier is an input of the round and the ring holds context written before it,
  // except the positions >= F - n_guard that this round's catch-up may store: a first
  // context block entirely older than that is fetched before waiting for the previous
  // kernel (the head post-processing, which writes Q and the block's keys/values).
  const AttGeom g = att_geom(a, b, split);
  const bool do_block = split == a.n_splits - 1;

  const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q);
  const __nv_bfloat16 *ring_k = static_cast<const __nv_bfloat16 *>(a.ring_k);
  const __nv_bfloat16 *ring_v = static_cast<const __nv_bfloat16 *>(a.ring_v);
  const __nv_bfloat16 *blk_k = static_cast<const __nv_bfloat16 *>(a.blk_k);
  const __nv_bfloat16 *blk_v = static_cast<const __nv_bfloat16 *>(a.blk_v);
  constexpr int CPR = D / 8;  // 16-byte chunks per row

  // Each thread copies chunk ch of the rows r0, r0 + rstep, ...; the ring slot of a row
  // advances with it (one modulo per tile, then wrap-around by subtraction).
  const size_t ring_head = (static_cast<size_t>(b) * a.n_kv_heads + h) * static_cast<size_t>(a.cap);
  auto load_kv = [&](int buf, int k0) {
    constexpr int rstep = 128 / CPR;
    const int ch = tid % CPR, r0 = tid / CPR;
    int slot = static_cast<int>((static_cast<long long>(g.p_lo) + k0 + r0) % a.cap);
    for (int kr = r0; kr < kAttKeys; kr += rstep) {
      const bool valid = k0 + kr < g.k_end;
      const size_t off = valid ? (ring_head + slot) * D : 0;
      cp_async16(smem_u32(sK + (buf * kAttKeys + kr) * RS + ch * 8), ring_k + off + ch * 8, valid);
      cp_async16(smem_u32(sV + (buf * kAttKeys + kr) * RS + ch * 8), ring_v + off + ch * 8, valid);
      slot += rstep;
      while (slot >= a.cap) slot -= a.cap;
    }
  };
  // Block keys/values [Kh; Kl; Vh; Vl] (16 rows each, rows >= W zero) go into the K
  // buffer the context loop leaves free after its last block (buffer n_blocks & 1); they
  // are loaded while that last block is processed.
  auto load_block = [&](int buf) {  // F16: [K; V], 16 rows each
    __nv_bfloat16 *dstb = sK + buf * kAttKeys * RS;
    for (int c = tid; c < (F16 ? 2 : 4) * 16 * CPR; c += 128) {
      const int part = c / (16 * CPR), cc = c % (16 * CPR);
      const int j = cc / CPR, ch = cc % CPR;
      const bool valid = j < a.W;
      const __nv_bfloat16 *base = F16 ? (part == 0 ? blk_k : blk_v)
                                      : (part < 2 ? blk_k : blk_v) + ((part & 1) ? a.blk_lo : 0);
      const __nv_bfloat16 *src =
          base + ((static_cast<size_t>(b) * a.n_kv_heads + h) * a.W + (valid ? j : 0)) * D + ch * 8;
      cp_async16(smem_u32(dstb + (part * 16 + j) * RS + ch * 8), src, valid);
    }
  };

  // F16: the ring chunks this thread loaded into buffer `buf`, rewritten as fp16 (called
  // after its copies have landed and before the barrier that publishes the tile)
  auto convert_kv = [&](int buf) {
    for (int c = tid; c < kAttKeys * CPR; c += 128) {
      const int kr = c / CPR, ch = c % CPR;
      bf16x8_to_f16_inplace(sK + (buf * kAttKeys + kr) * RS + ch * 8);
      bf16x8_to_f16_inplace(sV + (buf * kAttKeys + kr) * RS + ch * 8);
    }
  };

  float o[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  const float sl2 = 1.4426950408889634f * rsqrtf(static_cast<float>(D));  // log2(e)/sqrt(D)

  const int g4 = lane >> 2, t4 = lane & 3;
  const int rowA = warp * 16 + g4, rowB = rowA + 8;
  const int iA = rowA % a.W, iB = rowB % a.W;
  const bool rvA = rowA < R, rvB = rowB < R;

  const int n_blocks = g.k_end > g.k_begin ? (g.k_end - g.k_begin + kAttKeys - 1) / kAttKeys : 0;
  const bool early = n_blocks > 0 && g.p_lo + g.k_begin + kAttKeys <= g.F - a.n_guard;
  if (early) {
    load_kv(0, g.k_begin);
    cp_async_commit();
  }
  pdl_wait();
  pdl_trigger();
  // Q tiles: row rr = g_head * W + i  <-  q[(b*W + i), (h*G + g_head)*D + d]
  for (int c = tid; c < (F16 ? 1 : 2) * kAttRows * CPR; c += 128) {
    const int part = c / (kAttRows * CPR), cc = c % (kAttRows * CPR);
    const int rr = cc / CPR, ch = cc % CPR;
    const bool valid = rr < R;
    const int gh = valid ? rr / a.W : 0, i = valid ? rr % a.W : 0;
    const __nv_bfloat16 *src = q + (part ? a.q_lo : 0) +
                               (static_cast<size_t>(b) * a.W + i) * a.n_q_heads * D +
                               (h * G + gh) * D + ch * 8;
    cp_async16(smem_u32(sQ + (part * kAttRows + rr) * RS + ch * 8), src, valid);
  }
  if (n_blocks > 0 && !early) load_kv(0, g.k_begin);
  else if (n_blocks == 0 && do_block) load_block(0);
  cp_async_commit();
  // the first context position every block row can see: keys from here on need no mask
  const long long p_all = a.window > 0 ? g.F + a.W - a.window : LLONG_MIN;
  cp_async_wait<0>();
  if (F16 && n_blocks > 0) convert_kv(0);
  __syncthreads();

  // A fragments of Q (hi or lo) for k-step ks
  auto q_frag = [&](int part, int ks, uint32_t (&f)[4]) {
    const int mi = lane >> 3;
    const int row = warp * 16 + (mi & 1) * 8 + (lane & 7);
    const int col = ks * 16 + (mi >> 1) * 8;
    ldsm_x4(smem_u32(sQ + (part * kAttRows + row) * RS + col), f[0], f[1], f[2], f[3]);
  };

  for (int blk = 0; blk < n_blocks; ++blk) {
    const int buf = blk & 1;
    const int k0 = g.k_begin + blk * kAttKeys;
    if (blk + 1 < n_blocks) load_kv(buf ^ 1, k0 + kAttKeys);
    else if (do_block) load_block(buf ^ 1);
    cp_async_commit();

    // S = (Qh + Ql) K^T for 16 rows x 64 keys
    float s[kAttKeys / 8][4];
#pragma unroll
    for (int nt = 0; nt < kAttKeys / 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t qh[4], ql[4];
      q_frag(0, ks, qh);
      if (!F16) q_frag(1, ks, ql);
#pragma unroll
      for (int nt = 0; nt < kAttKeys / 8; nt += 2) {
        const int mi = lane >> 3;
        const int key = (nt + (mi >> 1)) * 8 + (lane & 7);
        const int col = ks * 16 + (mi & 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_u32(sK + (buf * kAttKeys + key) * RS + col), b0, b1, b2, b3);
        if constexpr (F16) {
          mma16816_f16(s[nt], qh, b0, b1);
          mma16816_f16(s[nt + 1], qh, b2, b3);
        } else {
          mma16816(s[nt], qh, b0, b1);
          mma16816(s[nt + 1], qh, b2, b3);
          mma16816(s[nt], ql, b0, b1);
          mma16816(s[nt + 1], ql, b2, b3);
        }
      }
    }
    if (k0 + kAttKeys <= g.k_end && g.p_lo + k0 >= p_all) {  // every key visible to every row
#pragma unroll
      for (int nt = 0; nt < kAttKeys / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nt][e] *= sl2;
    } else {
#pragma unroll
      for (int nt = 0; nt < kAttKeys / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int k = k0 + nt * 8 + 2 * t4 + (e & 1);
          const bool top = e < 2;
          const bool vis = (top ? rvA : rvB) && ctx_visible(a, g, top ? iA : iB, k);
          s[nt][e] = vis ? s[nt][e] * sl2 : -INFINITY;
        }
    }
    float alpha[2];
    softmax_update<kAttKeys / 8>(s, m_run, l_run, alpha);
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      o[n][0] *= alpha[0];
      o[n][1] *= alpha[0];
      o[n][2] *= alpha[1];
      o[n][3] *= alpha[1];
    }
    // O += (Ph + Pl) V
#pragma unroll
    for (int kk = 0; kk < kAttKeys / 16; ++kk) {
      uint32_t ph[4], pl[4];
      if constexpr (F16) {
        ph[0] = pack_f16(s[2 * kk][0], s[2 * kk][1]);
        ph[1] = pack_f16(s[2 * kk][2], s[2 * kk][3]);
        ph[2] = pack_f16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        ph[3] = pack_f16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
      } else {
        split_pack(s[2 * kk][0], s[2 * kk][1], ph[0], pl[0]);
        split_pack(s[2 * kk][2], s[2 * kk][3], ph[1], pl[1]);
        split_pack(s[2 * kk + 1][0], s[2 * kk + 1][1], ph[2], pl[2]);
        split_pack(s[2 * kk + 1][2], s[2 * kk + 1][3], ph[3], pl[3]);
      }
#pragma unroll
      for (int nd = 0; nd < D / 8; nd += 2) {
        const int mi = lane >> 3;
        const int key = kk * 16 + (mi & 1) * 8 + (lane & 7);
        const int col = (nd + (mi >> 1)) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_u32(sV + (buf * kAttKeys + key) * RS + col), b0, b1, b2, b3);
        if constexpr (F16) {
          mma16816_f16(o[nd], ph, b0, b1);
          mma16816_f16(o[nd + 1], ph, b2, b3);
        } else {
          mma16816(o[nd], ph, b0, b1);
          mma16816(o[nd + 1], ph, b2, b3);
          mma16816(o[nd], pl, b0, b1);
          mma16816(o[nd + 1], pl, b2, b3);
        }
      }
    }
    cp_async_wait<0>();
    if (F16 && blk + 1 < n_blocks) convert_kv(buf ^ 1);
    __syncthreads();
  }

  if (do_block) {
    if (n_blocks == 0) {  // the block tile was loaded with Q; nothing else is in flight
      cp_async_wait<0>();
      __syncthreads();
    }
    // [Kh; Kl; Vh; Vl] (F16: [K; V]), 16 rows each
    const __nv_bfloat16 *sB = sK + (n_blocks & 1) * kAttKeys * RS;
    constexpr int kV = F16 ? 1 : 2;  // first V part
    // S = Qh Kh + Ql Kh + Qh Kl over the (up to) 16 block keys (F16: Q K)
    float s[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t qh[4], ql[4];
      q_frag(0, ks, qh);
      const int mi = lane >> 3;
      const int key = (mi >> 1) * 8 + (lane & 7);
      const int col = ks * 16 + (mi & 1) * 8;
      uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
      ldsm_x4(smem_u32(sB + (0 * 16 + key) * RS + col), h0, h1, h2, h3);
      if constexpr (F16) {
        mma16816_f16(s[0], qh, h0, h1);
        mma16816_f16(s[1], qh, h2, h3);
      } else {
        q_frag(1, ks, ql);
        ldsm_x4(smem_u32(sB + (1 * 16 + key) * RS + col), l0, l1, l2, l3);
        mma16816(s[0], qh, h0, h1);
        mma16816(s[1], qh, h2, h3);
        mma16816(s[0], ql, h0, h1);
        mma16816(s[1], ql, h2, h3);
        mma16816(s[0], qh, l0, l1);
        mma16816(s[1], qh, l2, l3);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = nt * 8 + 2 * t4 + (e & 1);
        const bool top = e < 2;
        const bool vis = (top ? rvA : rvB) && blk_visible(a, top ? iA : iB, j);
        s[nt][e] = vis ? s[nt][e] * sl2 : -INFINITY;
      }
    float alpha[2];
    softmax_update<2>(s, m_run, l_run, alpha);
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      o[n][0] *= alpha[0];
      o[n][1] *= alpha[0];
      o[n][2] *= alpha[1];
      o[n][3] *= alpha[1];
    }
    uint32_t ph[4], pl[4];
    if constexpr (F16) {
      ph[0] = pack_f16(s[0][0], s[0][1]);
      ph[1] = pack_f16(s[0][2], s[0][3]);
      ph[2] = pack_f16(s[1][0], s[1][1]);
      ph[3] = pack_f16(s[1][2], s[1][3]);
    } else {
      split_pack(s[0][0], s[0][1], ph[0], pl[0]);
      split_pack(s[0][2], s[0][3], ph[1], pl[1]);
      split_pack(s[1][0], s[1][1], ph[2], pl[2]);
      split_pack(s[1][2], s[1][3], ph[3], pl[3]);
    }
#pragma unroll
    for (int nd = 0; nd < D / 8; nd += 2) {
      const int mi = lane >> 3;
      const int key = (mi & 1) * 8 + (lane & 7);
      const int col = (nd + (mi >> 1)) * 8;
      uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
      ldsm_x4_t(smem_u32(sB + (kV * 16 + key) * RS + col), h0, h1, h2, h3);
      if constexpr (F16) {
        mma16816_f16(o[nd], ph, h0, h1);
        mma16816_f16(o[nd + 1], ph, h2, h3);
      } else {
        ldsm_x4_t(smem_u32(sB + (3 * 16 + key) * RS + col), l0, l1, l2, l3);
        mma16816(o[nd], ph, h0, h1);
        mma16816(o[nd + 1], ph, h2, h3);
        mma16816(o[nd], pl, h0, h1);
        mma16816(o[nd + 1], pl, h2, h3);
        mma16816(o[nd], ph, l0, l1);
        mma16816(o[nd + 1], ph, l2, l3);
      }
    }
  }

  // ---- partial outputs
  const size_t bh = static_cast<size_t>(b) * a.n_kv_heads + h;
  float *po = a.part_o + (bh * a.n_splits + split) * kAttRows * D;
  float2 *pml = a.part_ml + (bh * a.n_splits + split) * kAttRows;
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    const int col = n * 8 + 2 * t4;
    *reinterpret_cast<float2 *>(po + rowA * D + col) = make_float2(o[n][0], o[n][1]);
    *reinterpret_cast<float2 *>(po + rowB * D + col) = make_float2(o[n][2], o[n][3]);
  }
  if (t4 == 0) {
    pml[rowA] = make_float2(m_run[0], l_run[0]);
    pml[rowB] = make_float2(m_run[1], l_run[1]);
  }

  // ---- merge the splits in this launch: every split of (b, h) counts itself once its
  // partial is stored, waits (bounded) for the others, then merges its share of the rows.
  // A launch has at most two CTAs per SM and never more than two per SM of the GPU, so all
  // splits are resident together; each stores its partial before it waits.
  __shared__ int s_abort;
  unsigned *arrived = a.counters + bh;
  unsigned *done = a.counters + static_cast<size_t>(a.B) * a.n_kv_heads + bh;
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    atomicAdd(arrived, 1u);
    s_abort = wait_count(arrived, static_cast<unsigned>(a.n_splits), kWaitLimitNs, 0) ? 0 : 1;
  }
  __syncthreads();
  if (s_abort) return;
  const int rp = (R + a.n_splits - 1) / a.n_splits;
  __shared__ float red[4][D + 4];
  if (a.n_splits <= kFewSplits)
    combine_rows_few<__nv_bfloat16, D, kFewSplits, 2>(a, b, h, min(R, split * rp),
                                                      min(R, (split + 1) * rp), warp, lane);
  else
    combine_rows<__nv_bfloat16, D>(a, b, h, min(R, split * rp), min(R, (split + 1) * rp), warp, lane,
                                   red);
  __syncthreads();
  if (tid == 0 && atomicAdd(done, 1u) == static_cast<unsigned>(a.n_splits - 1)) {
    *arrived = 0u;  // every split is past its wait: ready for the next launch
    *done = 0u;
  }
}

// fp32 path (small geometries): one CTA per (query head, request), exact fp32 softmax.
__global__ void __launch_bounds__(128) attention_f32_kernel(const __grid_constant__ AttArgs a) {
  extern __shared__ float sc[];  // [n_keys_max]
  const int qh = blockIdx.x, b = blockIdx.y;
  const int G = a.n_q_heads / a.n_kv_heads;
  const int h = qh / G;
  const int D = a.head_dim;
  pdl_wait();
  pdl_trigger();
  AttGeom g = att_geom(a, b, 0);
  g.k_begin = 0;
  g.k_end = g.n_ctx;
  const int n_keys = g.n_ctx + a.W;
  const float *q = static_cast<const float *>(a.q);
  const float *rk = static_cast<const float *>(a.ring_k);
  const float *rv = static_cast<const float *>(a.ring_v);
  const float *bk = static_cast<const float *>(a.blk_k);
  const float *bvv = static_cast<const float *>(a.blk_v);
  __shared__ float red[32];
  const float scale = rsqrtf(static_cast<float>(D));
  auto key_ptr = [&](int k, bool val) -> const float * {
    if (k < g.n_ctx) {
      const long long p = g.p_lo + k;
      return (val ? rv : rk) + ((static_cast<size_t>(b) * a.n_kv_heads + h) * a.cap + p % a.cap) * D;
    }
    return (val ? bvv : bk) + ((static_cast<size_t>(b) * a.n_kv_heads + h) * a.W + (k - g.n_ctx)) * D;
  };
  for (int i = 0; i < a.W; ++i) {
    const float *qi = q + (static_cast<size_t>(b) * a.W + i) * a.n_q_heads * D + qh * D;
    float lmax = -INFINITY;
    for (int k = threadIdx.x; k < n_keys; k += blockDim.x) {
      float sdot = -INFINITY;
      if (k < g.n_ctx ? ctx_visible(a, g, i, k) : blk_visible(a, i, k - g.n_ctx)) {
        const float *kp = key_ptr(k, false);
        float acc = 0.f;
        for (int d = 0; d < D; ++d) acc += qi[d] * kp[d];
        sdot = acc * scale;
      }
      sc[k] = sdot;
      lmax = fmaxf(lmax, sdot);
    }
    lmax = warp_max(lmax);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = lmax;
    __syncthreads();
    float M = -INFINITY;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) M = fmaxf(M, red[w]);
    __syncthreads();
    float lsum = 0.f;
    for (int k = threadIdx.x; k < n_keys; k += blockDim.x) {
      const float e = sc[k] == -INFINITY ? 0.f : expf(sc[k] - M);
      sc[k] = e;
      lsum += e;
    }
    lsum = warp_sum(lsum);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = lsum;
    __syncthreads();
    float L = 0.f;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) L += red[w];
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
      float acc = 0.f;
      for (int k = 0; k < n_keys; ++k)
        if (sc[k] != 0.f) acc += sc[k] * key_ptr(k, true)[d];
      float *out = static_cast<float *>(a.out) +
                   (static_cast<size_t>(b) * a.W + i) * a.n_q_heads * D + qh * D;
      out[d] = acc / L;
    }
    __syncthreads();
  }
}

size_t attention_smem_bytes(int head_dim) {
  return static_cast<size_t>(2 * kAttRows + 4 * kAttKeys) * (head_dim + kAttPad) * 2;
}
size_t attention_partial_floats(int B, int n_kv_heads, int n_splits, int head_dim) {
  return static_cast<size_t>(B) * n_kv_heads * n_splits * kAttRows * head_dim;
}
size_t attention_ml_count(int B, int n_kv_heads, int n_splits) {
  return static_cast<size_t>(B) * n_kv_heads * n_splits * kAttRows;
}
int attention_rows_max() { return kAttRows; }

std::string launch_attention(const AttArgs &a, int dtype, cudaStream_t stream) {
  cudaError_t e;
  if (dtype == 1) {
    const size_t smem = static_cast<size_t>(a.max_keys) * sizeof(float);
    static bool set = false;
    if (!set) {
      cudaFuncSetAttribute(attention_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           200 * 1024);
      set = true;
    }
    e = launch_pdl(attention_f32_kernel, dim3(a.n_q_heads, a.B), dim3(128), smem, stream, a);
    if (e != cudaSuccess) return std::string("attention launch: ") + cudaGetErrorString(e);
    return {};
  }
  const size_t smem = attention_smem_bytes(a.head_dim);
  auto go = [&](auto kernel) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    return launch_pdl(kernel, dim3(a.n_splits, a.n_kv_heads, a.B), dim3(128), smem, stream, a);
  };
  if (a.head_dim == 128)
    e = a.f16 ? go(attention_bf16_kernel<128, true>) : go(attention_bf16_kernel<128, false>);
  else
    e = a.f16 ? go(attention_bf16_kernel<64, true>) : go(attention_bf16_kernel<64, false>);
  if (e != cudaSuccess) return std::string("attention launch: ") + cudaGetErrorString(e);
  return {};
}

}  // namespace bd
