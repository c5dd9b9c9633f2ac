// Fused DSpine bridge ("DSpine for Qwen3.8-27B: Causal Features Through Depth", section
// "The bridge: read 1,024 features, write through rank 512"; "DSpine 完全拆解", sections on
// adjacent causal injection, gating and write-back).  For T = B*W <= 32 rows the
// bridge's three products stream only 19 MB of weights at the 27B size, and as five
// separate launches (row norm, code read, code, gate maps + message, write) its time was
// dominated by launch boundaries, dependency waits and split-tile reductions.  Here one
// launch of one CTA per SM runs it in four phases separated by grid-wide barriers:
//   P1  z'_q = R_l[:, K_q] x[:, K_q] per K chunk q, and the chunk's sums of squares of x
//   P2  z' = sum_q z'_q (fixed order), r_t = RMS(x_t), |z'|^2 partial sums per row group
//   P3  [G; G_p; A] z', scaled per token into the products of the codes
//       c_t = sqrt(Rc) z'_t / (|z'_t| + eps (r_t + eps)) (the code of x_t / (r_t + eps);
//       anchors sqrt(Rc) C[a]); g = sigmoid(G c_t + G_p c_{t-1} + b), m_t = g * (A c_{t-1}),
//       m_0 = 0; the tail export of the last layer
//   P4  x_t += r_t W_l m_t for every row but the anchor
// The products run on mma.sync across the CTA's 8 warps with the packed image's fp16
// weights and fp16 activations (the row chunks, codes and messages): at these shapes
// (N <= 32 token columns, short K per CTA) the warps' tensor instructions finish each
// product in a few microseconds without a TMEM round trip.  Weights come from the packed
// image, whose boxes are in the 128-byte-swizzled order (conflict-free ldmatrix): the
// first phase's as bulk copies issued before the dependency wait, P4's once the CTA's
// earlier product is done with that area.  The activations (x, the codes, the message)
// are written in the same swizzled box order, so the codes and the message reach shared
// memory as single bulk copies.  Partial sums are added in a fixed order, so results are
// deterministic.  Every CTA is resident at once (grid = SM count, one CTA per SM), each
// wait is bounded (wait_count, mbar_wait), and a wait that gives up ends the launch with
// the error word set.
#include "bd_device.cuh"
#include "bd_internal.h"
#include "bd_kernels.h"

#include <algorithm>

namespace bd {

BD_DEFINE_ERROR_TAKER(take_error_word_bridge)

constexpr int kBrThreads = 256;  // 8 warps
constexpr int kBrMaxKz = 32;     // K chunks of the code read (P1), at most
constexpr int kW4Rows = 32;      // rows of W_l per P4 item
// Block rows of one launch (B * W).  The phases are written for any multiple of 16 rows up
// to 128, but at B * W = 128 (27B geometry) one launch measured slower than the separate
// products (a 1588 against a 1560 us step): its code read stages 128 rows of fp32 residual
// per CTA and its gate phase runs on only Mc / 16 CTAs.
constexpr int kBrMaxT = 32;
constexpr int kBrMaxJ = 4;       // float4 columns per lane of a P1 chunk row: kz <= 512
constexpr int kBrMaxGz = 16;     // 128-row groups of the code: Rc <= 2048
constexpr int kP3Stride = 6144;  // bytes per K box of the P3 weights: G, G_p, A slices of 16 rows
constexpr int kP4Stride = 8192;  // bytes per K box of the P4 weights: two 32-row items

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
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
// A fragment (16 rows x 16 k) of a weight slice in the packed image's order: rows of 128
// bytes (64 fp16 of one K box), 16-byte chunk c of row r stored at chunk c ^ (r % 8); the
// slice starts at a row that is a multiple of 8.  kc: which 16 columns of the box.
__device__ __forceinline__ void ld_a(const uint8_t *box, int row0, int kc, uint32_t (&A)[4]) {
  const int lane = threadIdx.x & 31, mi = lane >> 3, ri = lane & 7;
  const int row = row0 + ri + 8 * (mi & 1), chunk = 2 * kc + (mi >> 1);
  ldsm4(smem_u32(box) + row * 128 + ((chunk ^ (row & 7)) << 4), A[0], A[1], A[2], A[3]);
}

// Activations as the MMA's B operand: R token rows x K, stored as K boxes of 64 columns,
// each box R rows of 128 bytes with the 16-byte chunk c of row r at chunk c ^ (r % 8) (the
// packed weights' swizzle).  Element offset:
__device__ __forceinline__ int act_off(int R, int r, int k) {
  return (k >> 6) * (R * 64) + r * 64 + ((((k & 63) >> 3) ^ (r & 7)) << 3) + (k & 7);
}
// B fragments of two 8-token n-tiles (tokens n0 .. n0+7 and n0+8 .. n0+15) x 16 k (k a
// multiple of 16): b0, b1 of the first, then of the second.
template <int R>
__device__ __forceinline__ void ld_b2(const __half *sx, int n0, int k, uint32_t (&Bf)[4]) {
  const int lane = threadIdx.x & 31, mi = lane >> 3, ri = lane & 7;
  const int row = n0 + (mi >> 1) * 8 + ri;
  ldsm4(smem_u32(sx + act_off(R, row, k + 8 * (mi & 1))), Bf[0], Bf[1], Bf[2], Bf[3]);
}

// fp16 activation stores (four values: one 8-byte store); a value beyond fp16's range
// sets the range error instead of passing as inf.
__device__ __forceinline__ void put4(__half *dst, float4 v) {
  flag_f16_range(f16_out_of_range(v.x) || f16_out_of_range(v.y) || f16_out_of_range(v.z) ||
                 f16_out_of_range(v.w));
  const __half2 h0 = __floats2half2_rn(v.x, v.y), h1 = __floats2half2_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t *>(&h0);
  u.y = *reinterpret_cast<const uint32_t *>(&h1);
  *reinterpret_cast<uint2 *>(dst) = u;
}
__device__ __forceinline__ void put1(__half *dst, float v) {
  flag_f16_range(f16_out_of_range(v));
  *dst = __float2half_rn(v);
}

// Grid-wide barrier on a counter that starts at zero: every CTA's writes before it are
// visible to every CTA after it (release arrival, acquire polling).  False if the wait gave
// up (error word set).
__device__ __forceinline__ bool grid_sync(unsigned *bar, int *s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(bar) : "memory");
    *s_ok = wait_count(bar, gridDim.x, kWaitLimitNs, 0) ? 1 : 0;
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

// Every thread waits (bounded) for the phase; the CTA agrees on the outcome.
__device__ __forceinline__ bool cta_wait(uint64_t *bar, uint32_t parity) {
  return __syncthreads_and(mbar_wait(bar, parity) ? 1 : 0) != 0;
}

template <int NT>
__global__ void __launch_bounds__(kBrThreads, 1) bridge_kernel(const __grid_constant__ BridgeArgs a) {
  constexpr int NTOK = NT * 8;             // token rows of the activation boxes
  constexpr int NP = NT / 2;               // pairs of 8-token n-tiles
  constexpr int NKS3 = 8 / NP;             // P3: warps per token pair, each a K share
  constexpr int P4P = NP >= 4 ? NP / 4 : 1;       // P4: token pairs per warp
  constexpr int NKS4 = NP >= 4 ? 1 : 4 / NP;      // P4: K shares of a token pair
  constexpr uint32_t kBoxB = NTOK * 128;   // bytes of one 64-column activation box
  extern __shared__ __align__(1024) uint8_t br_smem[];
  // shared-memory areas: P1 uses [R chunk | x chunk], P3 [weight slices | code chunk | ...
  // sums], P4 [message | W_l rows | sums]; an area is refilled only after its phase is done
  uint8_t *sw = br_smem;                              // P1 / P3 weights, P4 message boxes
  __half *sx1 = reinterpret_cast<__half *>(br_smem + a.off_x);
  uint8_t *sc3 = br_smem + a.off_c;
  uint8_t *sw4 = br_smem + a.off_w4;
  float *sred = reinterpret_cast<float *>(br_smem + a.off_red);
  // 0: first weights, 1: P4 weights, 2: P3 codes, 3: P4 message
  __shared__ __align__(8) uint64_t mb[4];
  __shared__ float red[kBrThreads / 32];
  __shared__ float s_scale[kBrMaxT];
  __shared__ int s_ok;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g4 = lane >> 2, t4 = lane & 3;
  const int T = a.T, H = a.H, Rc = a.Rc, Mc = a.Mc, W = a.W, cta = blockIdx.x;
  const int nbh = H / 64, nbc = Rc / 64, nbm = Mc / 64, gz = (Rc + 127) / 128;
  const bool in_p1 = cta < a.n1, in_p3 = cta >= a.n1 && cta < a.n1 + a.n3;
  const int n4 = H / kW4Rows;
  const int my4 = cta < n4 ? (n4 - 1 - cta) / static_cast<int>(gridDim.x) + 1 : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(&mb[i], 1);
    fence_barrier_init();
  }
  __syncthreads();

  // P4's rows of W_l (item it, box b at b * kP4Stride + it * 4096), thread 0
  auto load_w4 = [&]() {
    if (my4 == 0) return;
    const uint64_t pol = policy_evict_first();
    mbar_arrive_expect_tx(&mb[1], static_cast<uint32_t>(my4 * nbm * 4096));
    for (int it = 0; it < my4; ++it) {
      const int p = cta + it * static_cast<int>(gridDim.x);
      const int tw = p * kW4Rows / 128, ro = p * kW4Rows % 128;
      for (int b = 0; b < nbm; ++b)
        bulk_load(sw4 + b * kP4Stride + it * 4096,
                  a.pk_w + (static_cast<size_t>(tw) * nbm + b) * kPackBox + ro * 128, 4096, &mb[1],
                  pol);
    }
  };
  // ---- weights of the first phase: bulk copies from the packed image (no earlier kernel
  // writes it, so they start before the dependency wait)
  if (threadIdx.x == 0) {
    const uint64_t pol = policy_evict_first();
    if (in_p1) {
      const int gi = cta / a.n_kz, q = cta % a.n_kz;
      const int nb = min(a.kz, H - q * a.kz) / 64;
      mbar_arrive_expect_tx(&mb[0], static_cast<uint32_t>(nb * kPackBox));
      bulk_load(sw, a.pk_r + (static_cast<size_t>(gi) * nbh + static_cast<size_t>(q) * (a.kz / 64)) * kPackBox,
                static_cast<uint32_t>(nb * kPackBox), &mb[0], pol);
    } else if (in_p3) {
      const int row0 = (cta - a.n1) * 16, tj = row0 / 128, ro = row0 % 128;
      mbar_arrive_expect_tx(&mb[0], static_cast<uint32_t>(3 * nbc * 2048));
      const uint8_t *img[3] = {a.pk_g, a.pk_gp, a.pk_a};
      for (int b = 0; b < nbc; ++b)
        for (int mat = 0; mat < 3; ++mat)
          bulk_load(sw + b * kP3Stride + mat * 2048,
                    img[mat] + (static_cast<size_t>(tj) * nbc + b) * kPackBox + ro * 128, 2048,
                    &mb[0], pol);
    } else {
      load_w4();
    }
  }
  bool w1_pending = in_p1 || in_p3, w4_pending = !in_p1 && !in_p3 && my4 > 0;

  auto body = [&]() -> void {
    pdl_wait();
    pdl_trigger();

    // ---- P1: code-read partials of K chunk q for the 128 rows of tile gi
    if (in_p1) {
      const int gi = cta / a.n_kz, q = cta % a.n_kz;
      const int k0 = q * a.kz, klen = min(a.kz, H - k0);
      // the chunk of every token row as fp16 (rows past T as zeros); row group 0 also
      // takes the rows' sums of squares and the tail export
      // (kRB rows of a warp at a time, every load of the batch issued before any is used)
      constexpr int kRB = NTOK / (kBrThreads / 32) < 4 ? NTOK / (kBrThreads / 32) : 4;
      for (int t0 = warp; t0 < NTOK; t0 += kRB * (kBrThreads / 32)) {
        float4 xv[kRB][kBrMaxJ];
#pragma unroll
        for (int u = 0; u < kRB; ++u)
#pragma unroll
          for (int jj = 0; jj < kBrMaxJ; ++jj) {
            const int t = t0 + u * (kBrThreads / 32), j = lane * 4 + jj * 128;
            xv[u][jj] = t < T && j < klen
                            ? __ldcg(reinterpret_cast<const float4 *>(a.x + static_cast<size_t>(t) * H + k0 + j))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
        for (int u = 0; u < kRB; ++u) {
          const int t = t0 + u * (kBrThreads / 32);
          float ss = 0.f;
#pragma unroll
          for (int jj = 0; jj < kBrMaxJ; ++jj) {
            const int j = lane * 4 + jj * 128;
            if (j >= klen) break;
            const float4 x4 = xv[u][jj];
            if (gi == 0 && a.tail && t < T)  // u: the pre-injection residual
              *reinterpret_cast<float4 *>(a.tail + static_cast<size_t>(t) * H + k0 + j) = x4;
            ss += x4.x * x4.x + x4.y * x4.y + x4.z * x4.z + x4.w * x4.w;
            put4(sx1 + act_off(NTOK, t, j), x4);
          }
          if (gi == 0 && t < T) {
            ss = warp_sum(ss);
            if (lane == 0) a.sspart[q * T + t] = ss;
          }
        }
      }
      w1_pending = false;
      if (!cta_wait(&mb[0], 0)) return;  // (its barrier also publishes the activation rows)
      const int r0 = warp * 16;
      float acc[NT][4] = {};
      if (gi * 128 + r0 < Rc) {
        for (int b = 0; b < klen / 64; ++b)
#pragma unroll
          for (int kc = 0; kc < 4; ++kc) {
            uint32_t A[4];
            ld_a(sw + b * kPackBox, r0, kc, A);
#pragma unroll
            for (int np = 0; np < NP; ++np) {
              uint32_t Bf[4];
              ld_b2<NTOK>(sx1, np * 16, b * 64 + kc * 16, Bf);
              mma_f16_16816(acc[2 * np], A, Bf[0], Bf[1]);
              mma_f16_16816(acc[2 * np + 1], A, Bf[2], Bf[3]);
            }
          }
      }
      __syncthreads();  // every warp is done with the weight and activation areas
      if (threadIdx.x == 0) {
        fence_proxy_async_shared();
        load_w4();
      }
      w4_pending = my4 > 0;
      if (gi * 128 + r0 < Rc) {
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
    if (!grid_sync(a.bar + 0, &s_ok)) return;

    // ---- P2: z' = the chunk sums in order, as fp16 activation boxes (the anchor rows:
    // their codebook rows); r; |z'|^2 per row group.  Each half of the CTA (128 threads,
    // one row each) takes one (token, row group) item per pass.
    for (int base = cta; base < T * gz; base += 2 * static_cast<int>(gridDim.x)) {
      const int h = threadIdx.x >> 7, lt = threadIdx.x & 127;
      const int it = base + h * static_cast<int>(gridDim.x);
      const bool valid = it < T * gz;
      const int t = valid ? it / gz : 0, gi = valid ? it % gz : 0;
      if (valid && gi == 0 && (lt >> 5) == 0) {  // the half's first warp: r_t
        float ss = 0.f;
        for (int q = lane; q < a.n_kz; q += 32) ss += __ldcg(a.sspart + q * T + t);
        ss = warp_sum(ss);
        if (lane == 0) {
          const float r = sqrtf(ss / H);
          a.r[t] = r;
          if (a.tail) a.tail[static_cast<size_t>(T) * H + t] = r;
        }
      }
      const int row = gi * 128 + lt;
      float z = 0.f;
      if (valid && row < Rc) {
        __half *zh = a.zc + act_off(NTOK, t, row);
        if (t % W == 0) {  // anchor: the code is sqrt(Rc) C[a], its scale applied after the product
          int an = a.anchors[t / W];
          if (an < 0 || an >= a.V) {
            atomicOr(&g_error_word, DEVERR_BAD_INDEX);
            an = 0;
          }
          put1(zh, __bfloat162float(a.codebook[static_cast<size_t>(an) * Rc + row]));
        } else {
          float pv[kBrMaxKz];
#pragma unroll
          for (int q = 0; q < kBrMaxKz; ++q)
            pv[q] = q < a.n_kz ? __ldcg(a.zpart + (static_cast<size_t>(q) * T + t) * Rc + row) : 0.f;
#pragma unroll
          for (int q = 0; q < kBrMaxKz; ++q) z += pv[q];
          put1(zh, z);
        }
      }
      // |z'|^2 of the half's item: its four warps' sums in order
      const float v = warp_sum(z * z);
      if (lane == 0) red[warp] = v;
      __syncthreads();
      if (lt == 0 && valid && t % W != 0)
        a.zsq[t * gz + gi] = ((red[4 * h] + red[4 * h + 1]) + red[4 * h + 2]) + red[4 * h + 3];
      __syncthreads();
    }
    if (!grid_sync(a.bar + 1, &s_ok)) return;

    // ---- P3: [G; G_p; A] z' for rows j0 .. j0+15, scaled per token into the products of
    // the codes c_t = s_t z'_t; gate maps and message.  Warp w takes token pair w % NP
    // (16 columns) and the K steps w / NP, w / NP + NKS3, ...
    if (in_p3) {
      const int j0 = (cta - a.n1) * 16;
      // the code boxes in chunks of p3_boxes (rows T .. NTOK-1 hold stale values; they
      // only reach accumulator columns that are never read)
      const uint8_t *zc = reinterpret_cast<const uint8_t *>(a.zc);
      auto load_codes = [&](int b0) {  // thread 0
        const int nb = min(a.p3_boxes, nbc - b0);
        fence_proxy_async_global();
        fence_proxy_async_shared();
        mbar_arrive_expect_tx(&mb[2], static_cast<uint32_t>(nb) * kBoxB);
        bulk_load(sc3, zc + static_cast<size_t>(b0) * kBoxB, static_cast<uint32_t>(nb) * kBoxB, &mb[2],
                  policy_evict_first());
      };
      if (threadIdx.x == 0) load_codes(0);
      if (threadIdx.x < T) {
        const int t = threadIdx.x;
        const float cs = sqrtf(static_cast<float>(Rc));
        if (t % W == 0) {
          s_scale[t] = cs;
        } else {
          float zq[kBrMaxGz];
#pragma unroll
          for (int gi = 0; gi < kBrMaxGz; ++gi) zq[gi] = gi < gz ? __ldcg(a.zsq + t * gz + gi) : 0.f;
          float zz = 0.f;
#pragma unroll
          for (int gi = 0; gi < kBrMaxGz; ++gi) zz += zq[gi];
          s_scale[t] = cs / (sqrtf(zz) + a.eps * (__ldcg(a.r + t) + a.eps));
        }
      }
      w1_pending = false;
      const bool ok_w = cta_wait(&mb[0], 0);  // (a failure returns once the codes have landed)
      const __half *sx = reinterpret_cast<const __half *>(sc3);
      const int tp = warp % NP, ks0 = warp / NP;
      float acc[3][2][4] = {};
      for (int b0 = 0, ch = 0; b0 < nbc; b0 += a.p3_boxes, ++ch) {
        const int nb = min(a.p3_boxes, nbc - b0);
        if (ch > 0 && threadIdx.x == 0) load_codes(b0);
        const bool ok_c = cta_wait(&mb[2], static_cast<uint32_t>(ch) & 1u);
        if (!ok_w || !ok_c) return;
        for (int ks = ks0; ks < nb * 4; ks += NKS3) {
          const int b = b0 + ks / 4, kc = ks % 4;
          uint32_t A[3][4];
#pragma unroll
          for (int mat = 0; mat < 3; ++mat) ld_a(sw + b * kP3Stride + mat * 2048, 0, kc, A[mat]);
          uint32_t Bf[4];
          ld_b2<NTOK>(sx, tp * 16, ks * 16, Bf);
#pragma unroll
          for (int mat = 0; mat < 3; ++mat) {
            mma_f16_16816(acc[mat][0], A[mat], Bf[0], Bf[1]);
            mma_f16_16816(acc[mat][1], A[mat], Bf[2], Bf[3]);
          }
        }
        __syncthreads();  // the chunk's boxes (and, at the end, the weights) are free
      }
      // K-share partials [share][mat][16 rows][NTOK], added in share order and scaled
#pragma unroll
      for (int mat = 0; mat < 3; ++mat)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int row = g4 + (e >> 1) * 8, t = tp * 16 + nt * 8 + 2 * t4 + (e & 1);
            sred[((ks0 * 3 + mat) * 16 + row) * NTOK + t] = acc[mat][nt][e];
          }
      __syncthreads();
      auto pre = [&](int mat, int j, int t) {
        float v = 0.f;
#pragma unroll
        for (int k = 0; k < NKS3; ++k) v += sred[((k * 3 + mat) * 16 + j) * NTOK + t];
        return v * s_scale[t];
      };
      __half *m = a.m;
      for (int idx = threadIdx.x; idx < 16 * T; idx += kBrThreads) {
        const int t = idx % T, j = idx / T, jj = j0 + j;  // consecutive threads: consecutive t
        const float gc = pre(0, j, t);
        if (a.tail) a.tail[static_cast<size_t>(T) * H + T + static_cast<size_t>(t) * Mc + jj] = gc;  // G c_t
        float mv = 0.f;
        if (t % W != 0) {
          const float zg = gc + pre(1, j, t - 1) + (a.gate_bias ? __bfloat162float(a.gate_bias[jj]) : 0.f);
          const float g = 1.f / (1.f + expf(-zg));
          mv = g * pre(2, j, t - 1);
        }
        put1(m + act_off(NTOK, t, jj), mv);
      }
      // the weight and code areas are free since the chunk loop's last barrier: phase 4's
      // rows, issued now so that their copies overlap the grid barrier
      if (threadIdx.x == 0) {
        fence_proxy_async_shared();
        load_w4();
      }
      w4_pending = my4 > 0;
    }
    if (!grid_sync(a.bar + 2, &s_ok)) return;

    // ---- P4: x_t += r_t W_l m_t, 32 rows of W_l per item (item it, K box b at
    // b * kP4Stride + it * 4096); warp w: 16-row half w & 1 of the item, and of the four
    // warp pairs each takes P4P token pairs (NT >= 8) or a K share of one token pair
    if (my4 > 0) {
      if (threadIdx.x == 0) {
        fence_proxy_async_global();
        fence_proxy_async_shared();
        mbar_arrive_expect_tx(&mb[3], static_cast<uint32_t>(nbm) * kBoxB);
        bulk_load(sw, a.m, static_cast<uint32_t>(nbm) * kBoxB, &mb[3], policy_evict_first());
      }
      if (threadIdx.x < T) s_scale[threadIdx.x] = __ldcg(a.r + threadIdx.x);  // r_t (P3 is done)
      // the residual entries this thread updates, loaded while the copies land
      constexpr int kMaxUpd = 2 * kW4Rows * NTOK / kBrThreads;
      const int n_upd = my4 * kW4Rows * T;
      float xv[kMaxUpd];
#pragma unroll
      for (int u = 0; u < kMaxUpd; ++u) {
        const int idx = threadIdx.x + u * kBrThreads;
        const int it = idx / (kW4Rows * T), rem = idx % (kW4Rows * T);
        const int row = rem % kW4Rows, t = rem / kW4Rows;
        xv[u] = idx < n_upd ? __ldcg(a.x + static_cast<size_t>(t) * H +
                                     (cta + it * static_cast<int>(gridDim.x)) * kW4Rows + row)
                            : 0.f;
      }
      w4_pending = false;
      const bool ok_w = cta_wait(&mb[1], 0), ok_m = cta_wait(&mb[3], 0);
      if (!ok_w || !ok_m) return;
      const __half *sm = reinterpret_cast<const __half *>(sw);
      const int mt = warp & 1, grp = warp >> 1;
      const int tp0 = NP >= 4 ? grp * P4P : grp % NP, ks = NP >= 4 ? 0 : grp / NP;
      const int kw = Mc / NKS4;
      for (int it = 0; it < my4; ++it) {
        float acc[2 * P4P][4] = {};
        for (int s4 = 0; s4 < kw / 16; ++s4) {
          const int k = ks * kw + s4 * 16, b = k / 64, kc = (k % 64) / 16;
          uint32_t A[4];
          ld_a(sw4 + b * kP4Stride + it * 4096, mt * 16, kc, A);
#pragma unroll
          for (int p = 0; p < P4P; ++p) {
            uint32_t Bf[4];
            ld_b2<NTOK>(sm, (tp0 + p) * 16, k, Bf);
            mma_f16_16816(acc[2 * p], A, Bf[0], Bf[1]);
            mma_f16_16816(acc[2 * p + 1], A, Bf[2], Bf[3]);
          }
        }
#pragma unroll
        for (int nt = 0; nt < 2 * P4P; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int row = mt * 16 + g4 + (e >> 1) * 8, t = tp0 * 16 + nt * 8 + 2 * t4 + (e & 1);
            sred[((it * NKS4 + ks) * kW4Rows + row) * NTOK + t] = acc[nt][e];
          }
      }
      __syncthreads();
#pragma unroll
      for (int u = 0; u < kMaxUpd; ++u) {
        const int idx = threadIdx.x + u * kBrThreads;
        if (idx >= n_upd) break;
        const int it = idx / (kW4Rows * T), rem = idx % (kW4Rows * T);
        const int row = rem % kW4Rows, t = rem / kW4Rows;
        if (t % W == 0) continue;
        float v = 0.f;
#pragma unroll
        for (int q = 0; q < NKS4; ++q) v += sred[((it * NKS4 + q) * kW4Rows + row) * NTOK + t];
        a.x[static_cast<size_t>(t) * H + (cta + it * static_cast<int>(gridDim.x)) * kW4Rows + row] =
            xv[u] + s_scale[t] * v;
      }
    }
  };
  body();
  // copies still in flight after an early exit are waited for (bounded) before the CTA ends
  if (w1_pending) mbar_wait(&mb[0], 0);
  if (w4_pending) mbar_wait(&mb[1], 0);
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

// Token rows of the activation boxes for T block rows (the kernel's NT * 8).
static int bridge_ntok(int T) { return T <= 16 ? 16 : 32; }

BridgePlan bridge_plan(int dtype, int T, int H, int Rc, int Mc, int sms) {
  BridgePlan p = {};
  if (dtype != 0 || T < 1 || T > kBrMaxT || H % 64 || Rc % 64 || Mc % 64 || Rc < 64 || Mc < 64 ||
      Rc > 128 * kBrMaxGz)
    return p;
  const size_t ntok = bridge_ntok(T), box = ntok * 128;  // bytes of an activation box
  const int gz = (Rc + 127) / 128;
  p.n3 = Mc / 16;
  const int avail = sms - p.n3;
  if (avail < gz) return p;
  const int nz = std::min(std::min(avail / gz, kBrMaxKz), H / 64);
  p.kz = ((H + nz - 1) / nz + 63) / 64 * 64;
  if (p.kz > 128 * kBrMaxJ) return p;
  p.n_kz = (H + p.kz - 1) / p.kz;
  p.n1 = gz * p.n_kz;
  const int n4 = H / kW4Rows, it4 = (n4 + sms - 1) / sms;
  if (it4 > 2) return p;  // P4 holds two items per K box
  const int nbc = Rc / 64, nbm = Mc / 64;
  const int np = static_cast<int>(ntok / 16), nks3 = 8 / np, nks4 = np >= 4 ? 1 : 4 / np;
  auto up = [](size_t v) { return (v + 1023) / 1024 * 1024; };
  // P1: [R chunk | x chunk]; P3: [weight slices | code chunk]; P4: [message | W_l rows |
  // sums] (the P3 sums share P4's area)
  p.off_x = up(static_cast<size_t>(p.kz / 64) * kPackBox);
  p.off_c = up(static_cast<size_t>(nbc) * kP3Stride);
  p.off_w4 = up(static_cast<size_t>(nbm) * box);
  p.off_red = up(p.off_w4 + static_cast<size_t>(nbm) * kP4Stride);
  const size_t red3 = static_cast<size_t>(nks3) * 3 * 16 * ntok * 4;
  const size_t red4 = static_cast<size_t>(it4) * nks4 * kW4Rows * ntok * 4;
  const size_t p1 = p.off_x + static_cast<size_t>(p.kz / 64) * box;
  const size_t p4 = p.off_red + std::max(red3, red4);
  const int lim = max_dyn_smem() - 2048;  // the kernel's static shared memory and alignment
  // the code chunk: as many boxes as fit beside the weight slices
  const size_t room = static_cast<size_t>(lim) > p.off_c ? static_cast<size_t>(lim) - p.off_c : 0;
  p.p3_boxes = static_cast<int>(std::min(static_cast<size_t>(nbc), room / box));
  if (p.p3_boxes < 1) return p;
  const size_t p3 = p.off_c + static_cast<size_t>(p.p3_boxes) * box;
  p.smem = std::max(std::max(p1, p3), p4);
  p.ok = lim > 0 && p.smem <= static_cast<size_t>(lim);
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
  if (bridge_ntok(args.T) == 16)
    e = go(bridge_kernel<2>);
  else
    e = go(bridge_kernel<4>);
  return e == cudaSuccess ? std::string() : std::string("bridge: ") + cudaGetErrorString(e);
}

}  // namespace bd
