// Fused DSpine bridge for small blocks ("DSpine for Qwen3.8-27B: Causal Features Through
// Depth", section "The bridge: read 1,024 features, write through rank 512"; "DSpine 完全
// 拆解", sections on adjacent causal injection, gating and write-back).  With T = B*W <= 32
// rows the bridge's three products stream only 19 MB of weights at the 27B size, and as
// five separate launches (row norm, code read, code, gate maps + message, write) its time
// was dominated by launch boundaries, dependency waits and split-tile reductions.  Here one
// launch of one CTA per SM runs it in four phases separated by grid-wide barriers:
//   P1  z'_q = R_l[:, K_q] x[:, K_q] per K chunk q, and the chunk's sums of squares of x
//   P2  z' = sum_q z'_q (fixed order), r_t = RMS(x_t), |z'|^2 partial sums per row group
//   P3  c_t = sqrt(Rc) z'_t / (|z'_t| + eps (r_t + eps)), which is the code of
//       x_t / (r_t + eps); anchors sqrt(Rc) C[a]; [G; G_p; A] c;
//       g = sigmoid(G c_t + G_p c_{t-1} + b), m_t = g * (A c_{t-1}), m_0 = 0; the tail
//       export of the last layer
//   P5  x_t += r_t W_l m_t for every row but the anchor
// Every CTA's weights (its R_l chunk or its 16 rows of G, G_p and A, and its rows of W_l)
// come from the packed weight image as bulk copies issued before the dependency wait, so
// the 19 MB stream in while the previous kernel finishes and the first phase stages x.
// The products run on mma.sync with bf16 hi + lo activation pairs (~16 mantissa bits);
// partial sums are added in a fixed order, so results are deterministic.  Every CTA is
// resident at once (grid = SM count, one CTA per SM), each wait is bounded (wait_count,
// mbar_wait), and a wait that gives up ends the launch with the error word set.
#include "bd_device.cuh"
#include "bd_internal.h"
#include "bd_kernels.h"

#include <algorithm>

namespace bd {

BD_DEFINE_ERROR_TAKER(take_error_word_bridge)

constexpr int kBrThreads = 256;  // 8 warps
constexpr int kBrMaxKz = 32;     // K chunks of the code read (P1), at most
constexpr int kW5Rows = 32;      // rows of W_l per P5 item (two 16-row tiles x 4 K quarters)

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
      "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                      uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void cp16_cg(void *dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}

// A fragment (16 rows x 16 k) of a weight slice in the packed image's order: rows of 128
// bytes (64 bf16 of one K box), 16-byte chunk c of row r stored at chunk c ^ (r % 8); the
// slice starts at a row that is a multiple of 8.  kc: which 16 columns of the box.
__device__ __forceinline__ void ld_a(const uint8_t *box, int row0, int kc, uint32_t (&A)[4]) {
  const int lane = threadIdx.x & 31, mi = lane >> 3, ri = lane & 7;
  const int row = row0 + ri + 8 * (mi & 1), chunk = 2 * kc + (mi >> 1);
  ldsm4(smem_u32(box) + row * 128 + ((chunk ^ (row & 7)) << 4), A[0], A[1], A[2], A[3]);
}
// B fragments of 8 tokens x 16 k from staged activations [2][ntok][BS] (hi block, lo
// block): hi b0, hi b1, lo b0, lo b1.
__device__ __forceinline__ void ld_b(const __nv_bfloat16 *sx, int BS, int ntok, int n0, int k,
                                     uint32_t (&Bf)[4]) {
  const int lane = threadIdx.x & 31, mi = lane >> 3, ri = lane & 7;
  const __nv_bfloat16 *p = sx + static_cast<size_t>((mi >> 1) * ntok + n0 + ri) * BS + k + 8 * (mi & 1);
  ldsm4(smem_u32(p), Bf[0], Bf[1], Bf[2], Bf[3]);
}

// bf16 hi + lo pair of four values (8-byte stores)
__device__ __forceinline__ void split4(float4 v, __nv_bfloat16 *hi, __nv_bfloat16 *lo) {
  const __nv_bfloat162 h0 = __floats2bfloat162_rn(v.x, v.y), h1 = __floats2bfloat162_rn(v.z, v.w);
  const float2 f0 = __bfloat1622float2(h0), f1 = __bfloat1622float2(h1);
  const __nv_bfloat162 l0 = __floats2bfloat162_rn(v.x - f0.x, v.y - f0.y);
  const __nv_bfloat162 l1 = __floats2bfloat162_rn(v.z - f1.x, v.w - f1.y);
  uint2 uh, ul;
  uh.x = *reinterpret_cast<const uint32_t *>(&h0);
  uh.y = *reinterpret_cast<const uint32_t *>(&h1);
  ul.x = *reinterpret_cast<const uint32_t *>(&l0);
  ul.y = *reinterpret_cast<const uint32_t *>(&l1);
  *reinterpret_cast<uint2 *>(hi) = uh;
  *reinterpret_cast<uint2 *>(lo) = ul;
}
__device__ __forceinline__ void put_split(__nv_bfloat16 *p, size_t lo_off, float v) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  p[0] = h;
  p[lo_off] = __float2bfloat16_rn(v - __bfloat162float(h));
}

// Grid-wide barrier on a counter that starts at zero: every CTA's writes before it are
// visible to every CTA after it.  False if the wait gave up (error word set).
__device__ __forceinline__ bool grid_sync(unsigned *bar, int *s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(bar, 1u);
    *s_ok = wait_count(bar, gridDim.x) ? 1 : 0;
    __threadfence();
  }
  __syncthreads();
  return *s_ok != 0;
}

// Sum over the CTA in a fixed order (warp trees, then warps 0..7); every thread gets it.
__device__ __forceinline__ float block_sum(float v, float *red) {
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < kBrThreads / 32; ++w) s += red[w];
  __syncthreads();
  return s;
}

template <int NT>
__global__ void __launch_bounds__(kBrThreads, 1) bridge_kernel(const __grid_constant__ BridgeArgs a) {
  constexpr int NTOK = NT * 8;
  extern __shared__ __align__(1024) uint8_t br_smem[];
  uint8_t *s1 = br_smem;                // P1 / P3 weights, then the staged message of P5
  uint8_t *s5 = br_smem + a.s1_bytes;   // P5 weights
  uint8_t *sa = s5 + a.s5_bytes;        // staged activations, then cross-warp partial sums
  __shared__ __align__(8) uint64_t wbar[2];
  __shared__ float red[kBrThreads / 32];
  __shared__ float s_scale[32];
  __shared__ int s_ok;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g4 = lane >> 2, t4 = lane & 3;
  const int T = a.T, H = a.H, Rc = a.Rc, Mc = a.Mc, W = a.W, cta = blockIdx.x;
  const int nbh = H / 64, nbc = Rc / 64, nbm = Mc / 64, gz = (Rc + 127) / 128;
  const bool in_p1 = cta < a.n1, in_p3 = cta >= a.n1 && cta < a.n1 + a.n3;
  const int n5 = H / kW5Rows;
  const int my5 = cta < n5 ? (n5 - 1 - cta) / static_cast<int>(gridDim.x) + 1 : 0;

  // ---- weights: bulk copies from the packed image (no earlier kernel writes them)
  if (threadIdx.x == 0) {
    mbar_init(&wbar[0], 1);
    mbar_init(&wbar[1], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t pol = policy_evict_first();
    if (in_p1) {
      const int gi = cta / a.n_kz, q = cta % a.n_kz;
      const int nb = min(a.kz, H - q * a.kz) / 64;
      mbar_arrive_expect_tx(&wbar[0], static_cast<uint32_t>(nb * kPackBox));
      bulk_load(s1, a.pk_r + (static_cast<size_t>(gi) * nbh + static_cast<size_t>(q) * (a.kz / 64)) * kPackBox,
                static_cast<uint32_t>(nb * kPackBox), &wbar[0], pol);
    } else if (in_p3) {
      const int row0 = (cta - a.n1) * 16, tj = row0 / 128, ro = row0 % 128;
      mbar_arrive_expect_tx(&wbar[0], static_cast<uint32_t>(3 * nbc * 2048));
      const uint8_t *img[3] = {a.pk_g, a.pk_gp, a.pk_a};
      for (int mat = 0; mat < 3; ++mat)
        for (int b = 0; b < nbc; ++b)
          bulk_load(s1 + (mat * nbc + b) * 2048,
                    img[mat] + (static_cast<size_t>(tj) * nbc + b) * kPackBox + ro * 128, 2048,
                    &wbar[0], pol);
    }
    if (my5 > 0) {
      mbar_arrive_expect_tx(&wbar[1], static_cast<uint32_t>(my5 * nbm * 4096));
      for (int it = 0; it < my5; ++it) {
        const int p = cta + it * static_cast<int>(gridDim.x);
        const int tw = p * kW5Rows / 128, ro = p * kW5Rows % 128;
        for (int b = 0; b < nbm; ++b)
          bulk_load(s5 + (it * nbm + b) * 4096,
                    a.pk_w + (static_cast<size_t>(tw) * nbm + b) * kPackBox + ro * 128, 4096,
                    &wbar[1], pol);
      }
    }
  }
  bool w1_pending = in_p1 || in_p3, w5_pending = my5 > 0;
  // a CTA that leaves early first waits (bounded) for its copies still in flight
  auto leave = [&]() {
    if (w1_pending) mbar_wait(&wbar[0], 0);
    if (w5_pending) mbar_wait(&wbar[1], 0);
  };

  pdl_wait();
  pdl_trigger();

  // ---- P1: code-read partials of K chunk q for the 128 rows of tile gi
  if (in_p1) {
    const int gi = cta / a.n_kz, q = cta % a.n_kz;
    const int k0 = q * a.kz, klen = min(a.kz, H - k0), BS = klen + 8;
    __nv_bfloat16 *sx = reinterpret_cast<__nv_bfloat16 *>(sa);
    for (int t = warp; t < NTOK; t += kBrThreads / 32) {
      float ss = 0.f;
      for (int j = lane * 4; j < klen; j += 128) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < T) {
          v = __ldcg(reinterpret_cast<const float4 *>(a.x + static_cast<size_t>(t) * H + k0 + j));
          if (gi == 0 && a.tail)  // u: the pre-injection residual
            *reinterpret_cast<float4 *>(a.tail + static_cast<size_t>(t) * H + k0 + j) = v;
        }
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        split4(v, sx + t * BS + j, sx + (NTOK + t) * BS + j);
      }
      if (gi == 0 && t < T) {
        ss = warp_sum(ss);
        if (lane == 0) a.sspart[q * T + t] = ss;
      }
    }
    __syncthreads();
    w1_pending = false;
    if (!mbar_wait(&wbar[0], 0)) {
      leave();
      return;
    }
    const int r0 = warp * 16;
    if (gi * 128 + r0 < Rc) {
      float acc[NT][4] = {};
      for (int b = 0; b < klen / 64; ++b)
#pragma unroll
        for (int kc = 0; kc < 4; ++kc) {
          uint32_t A[4];
          ld_a(s1 + b * kPackBox, r0, kc, A);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            uint32_t Bf[4];
            ld_b(sx, BS, NTOK, nt * 8, b * 64 + kc * 16, Bf);
            mma_bf16_16816(acc[nt], A, Bf[0], Bf[1]);
            mma_bf16_16816(acc[nt], A, Bf[2], Bf[3]);
          }
        }
      float *zp = a.zpart + static_cast<size_t>(q) * T * Rc;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = gi * 128 + r0 + g4 + (e >> 1) * 8, t = nt * 8 + 2 * t4 + (e & 1);
          if (row < Rc && t < T) zp[static_cast<size_t>(t) * Rc + row] = acc[nt][e];
        }
    }
  }
  if (!grid_sync(a.bar + 0, &s_ok)) {
    leave();
    return;
  }

  // ---- P2: z' = the chunk sums in order; r; |z'|^2 per row group
  for (int it = cta; it < T * gz; it += gridDim.x) {
    const int t = it / gz, gi = it % gz;
    if (gi == 0 && warp == 0) {
      float ss = 0.f;
      for (int q = lane; q < a.n_kz; q += 32) ss += __ldcg(a.sspart + q * T + t);
      ss = warp_sum(ss);
      if (lane == 0) {
        const float r = sqrtf(ss / H);
        a.r[t] = r;
        if (a.tail) a.tail[static_cast<size_t>(T) * H + t] = r;
      }
    }
    if (t % W == 0) continue;  // the anchor's code comes from the codebook
    const int row = gi * 128 + threadIdx.x;
    float z = 0.f;
    if (threadIdx.x < 128 && row < Rc) {
      float v[kBrMaxKz];
#pragma unroll
      for (int q = 0; q < kBrMaxKz; ++q)
        v[q] = q < a.n_kz ? __ldcg(a.zpart + (static_cast<size_t>(q) * T + t) * Rc + row) : 0.f;
#pragma unroll
      for (int q = 0; q < kBrMaxKz; ++q) z += v[q];
      a.z[static_cast<size_t>(t) * Rc + row] = z;
    }
    const float zz = block_sum(z * z, red);
    if (threadIdx.x == 0) a.zsq[t * gz + gi] = zz;
  }
  if (!grid_sync(a.bar + 1, &s_ok)) {
    leave();
    return;
  }

  // ---- P3: codes, gate maps and message for rows j0 .. j0+15 of G, G_p, A
  if (in_p3) {
    const int j0 = (cta - a.n1) * 16;
    const float cs = sqrtf(static_cast<float>(Rc));
    if (threadIdx.x < T) {
      const int t = threadIdx.x;
      if (t % W == 0) {
        s_scale[t] = cs;
      } else {
        float zz = 0.f;
        for (int gi = 0; gi < gz; ++gi) zz += __ldcg(a.zsq + t * gz + gi);
        s_scale[t] = cs / (sqrtf(zz) + a.eps * (__ldcg(a.r + t) + a.eps));
      }
    }
    __syncthreads();
    w1_pending = false;
    if (!mbar_wait(&wbar[0], 0)) {
      leave();
      return;
    }
    __nv_bfloat16 *sx = reinterpret_cast<__nv_bfloat16 *>(sa);
    float acc[3][NT][4] = {};
    for (int k0 = 0; k0 < Rc; k0 += a.kc3) {
      const int klen = min(a.kc3, Rc - k0), BS = klen + 8, c4 = klen / 4;
      for (int idx = threadIdx.x; idx < NTOK * c4; idx += kBrThreads) {
        const int t = idx / c4, k = k0 + (idx % c4) * 4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < T) {
          const float s = s_scale[t];
          if (t % W == 0) {
            int an = a.anchors[t / W];
            if (an < 0 || an >= a.V) {
              atomicOr(&g_error_word, DEVERR_BAD_INDEX);
              an = 0;
            }
            const uint2 u = *reinterpret_cast<const uint2 *>(a.codebook + static_cast<size_t>(an) * Rc + k);
            const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
            const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
            v = make_float4(s * f0.x, s * f0.y, s * f1.x, s * f1.y);
          } else {
            v = __ldcg(reinterpret_cast<const float4 *>(a.z + static_cast<size_t>(t) * Rc + k));
            v = make_float4(s * v.x, s * v.y, s * v.z, s * v.w);
          }
        }
        split4(v, sx + t * BS + (k - k0), sx + (NTOK + t) * BS + (k - k0));
      }
      __syncthreads();
      for (int ks = warp; ks < klen / 16; ks += kBrThreads / 32) {
        const int k = k0 + ks * 16, b = k / 64, kc = (k % 64) / 16;
        uint32_t A[3][4];
#pragma unroll
        for (int mat = 0; mat < 3; ++mat) ld_a(s1 + (mat * nbc + b) * 2048, 0, kc, A[mat]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          uint32_t Bf[4];
          ld_b(sx, BS, NTOK, nt * 8, ks * 16, Bf);
#pragma unroll
          for (int mat = 0; mat < 3; ++mat) {
            mma_bf16_16816(acc[mat][nt], A[mat], Bf[0], Bf[1]);
            mma_bf16_16816(acc[mat][nt], A[mat], Bf[2], Bf[3]);
          }
        }
      }
      __syncthreads();
    }
    // per-warp K partials [warp][mat][16 rows][NTOK], added in warp order
    float *red3 = reinterpret_cast<float *>(sa);
#pragma unroll
    for (int mat = 0; mat < 3; ++mat)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = g4 + (e >> 1) * 8, t = nt * 8 + 2 * t4 + (e & 1);
          red3[((warp * 3 + mat) * 16 + row) * NTOK + t] = acc[mat][nt][e];
        }
    __syncthreads();
    auto pre = [&](int mat, int j, int t) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kBrThreads / 32; ++w) s += red3[((w * 3 + mat) * 16 + j) * NTOK + t];
      return s;
    };
    const size_t mlo = static_cast<size_t>(a.TP) * Mc;
    for (int idx = threadIdx.x; idx < 16 * T; idx += kBrThreads) {
      const int j = idx % 16, t = idx / 16, jj = j0 + j;
      const float gc = pre(0, j, t);
      if (a.tail) a.tail[static_cast<size_t>(T) * H + T + static_cast<size_t>(t) * Mc + jj] = gc;  // G c_t
      float mv = 0.f;
      if (t % W != 0) {
        const float zg = gc + pre(1, j, t - 1) + (a.gate_bias ? __bfloat162float(a.gate_bias[jj]) : 0.f);
        const float g = 1.f / (1.f + expf(-zg));
        mv = g * pre(2, j, t - 1);
      }
      put_split(a.m + static_cast<size_t>(t) * Mc + jj, mlo, mv);
    }
  }
  if (!grid_sync(a.bar + 2, &s_ok)) {
    leave();
    return;
  }

  // ---- P5: x_t += r_t W_l m_t, 32 rows of W_l per item
  if (my5 > 0) {
    const int BS = Mc + 8, c8 = Mc / 8;
    __nv_bfloat16 *sm = reinterpret_cast<__nv_bfloat16 *>(s1);
    for (int idx = threadIdx.x; idx < 2 * NTOK * c8; idx += kBrThreads) {
      const int part = idx / (NTOK * c8), rq = idx % (NTOK * c8), t = rq / c8, ch = rq % c8;
      const bool valid = t < T;
      const __nv_bfloat16 *src = a.m + static_cast<size_t>(part) * a.TP * Mc +
                                 static_cast<size_t>(valid ? t : 0) * Mc + ch * 8;
      cp16_cg(sm + (part * NTOK + t) * BS + ch * 8, src, valid);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    w5_pending = false;
    if (!mbar_wait(&wbar[1], 0)) return;
    const int mt = warp & 1, kq = warp >> 1, kw = Mc / 4;
    float *red5 = reinterpret_cast<float *>(sa);
    for (int it = 0; it < my5; ++it) {
      const int p = cta + it * static_cast<int>(gridDim.x);
      float acc[NT][4] = {};
      for (int s = 0; s < kw / 16; ++s) {
        const int k = kq * kw + s * 16, b = k / 64, kc = (k % 64) / 16;
        uint32_t A[4];
        ld_a(s5 + (it * nbm + b) * 4096, mt * 16, kc, A);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          uint32_t Bf[4];
          ld_b(sm, BS, NTOK, nt * 8, k, Bf);
          mma_bf16_16816(acc[nt], A, Bf[0], Bf[1]);
          mma_bf16_16816(acc[nt], A, Bf[2], Bf[3]);
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = mt * 16 + g4 + (e >> 1) * 8, t = nt * 8 + 2 * t4 + (e & 1);
          red5[(kq * kW5Rows + row) * NTOK + t] = acc[nt][e];
        }
      __syncthreads();
      for (int idx = threadIdx.x; idx < kW5Rows * T; idx += kBrThreads) {
        const int row = idx % kW5Rows, t = idx / kW5Rows;
        if (t % W == 0) continue;
        float s = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) s += red5[(q * kW5Rows + row) * NTOK + t];
        a.x[static_cast<size_t>(t) * H + p * kW5Rows + row] += __ldcg(a.r + t) * s;
      }
      __syncthreads();
    }
  }
}

// ------------------------------------------------------------------ host
static int max_dyn_smem() {
  static int v = -1;
  if (v < 0) {
    int dev = 0, optin = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      optin = 0;
    v = optin;
  }
  return v;
}

BridgePlan bridge_plan(int dtype, int T, int H, int Rc, int Mc, int sms) {
  BridgePlan p = {};
  if (dtype != 0 || T < 1 || T > 32 || H % 64 || Rc % 64 || Mc % 64 || Rc < 64 || Mc < 64) return p;
  const int ntok = T <= 16 ? 16 : 32;
  const int gz = (Rc + 127) / 128;
  p.n3 = Mc / 16;
  const int avail = sms - p.n3;
  if (avail < gz) return p;
  const int nz = std::min(std::min(avail / gz, kBrMaxKz), H / 64);
  p.kz = ((H + nz - 1) / nz + 63) / 64 * 64;
  p.n_kz = (H + p.kz - 1) / p.kz;
  p.n1 = gz * p.n_kz;
  const int n5 = H / kW5Rows, it5 = (n5 + sms - 1) / sms;
  const size_t act_p1 = static_cast<size_t>(4) * ntok * (p.kz + 8);
  const size_t red3 = static_cast<size_t>(8) * 3 * 16 * ntok * 4;
  const size_t red5 = static_cast<size_t>(4) * kW5Rows * ntok * 4;
  p.sa_bytes = std::max(act_p1, std::max(red3, red5));
  // P3 stages K in chunks that fit the activation area
  p.kc3 = std::min(Rc, static_cast<int>((p.sa_bytes / (4 * ntok) - 8) / 64 * 64));
  if (p.kc3 < 64) return p;
  p.s1_bytes = std::max(static_cast<size_t>(p.kz / 64) * kPackBox,
                        std::max(static_cast<size_t>(3) * (Rc / 64) * 2048,
                                 static_cast<size_t>(4) * ntok * (Mc + 8)));
  p.s1_bytes = (p.s1_bytes + 1023) / 1024 * 1024;
  p.s5_bytes = static_cast<size_t>(it5) * (Mc / 64) * 4096;
  p.smem = p.s1_bytes + p.s5_bytes + p.sa_bytes;
  const int lim = max_dyn_smem();
  p.ok = lim > 0 && p.smem + 1024 <= static_cast<size_t>(lim);
  return p;
}

std::string launch_bridge(const BridgeArgs &args, const BridgePlan &plan, int sms, cudaStream_t s) {
  cudaError_t e;
  auto go = [&](auto kernel) {
    cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(plan.smem));
    if (r != cudaSuccess) return r;
    return launch_pdl(kernel, dim3(sms), dim3(kBrThreads), plan.smem, s, args);
  };
  if (args.T <= 16)
    e = go(bridge_kernel<2>);
  else
    e = go(bridge_kernel<4>);
  return e == cudaSuccess ? std::string() : std::string("bridge: ") + cudaGetErrorString(e);
}

}  // namespace bd
