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
// bf16 path, on the 5th-generation tensor cores.  One CTA per (key split, KV head,
// request); all G = Hq/Hkv query heads of the KV head and all W block rows (G*W <= 64
// query rows) share every K/V tile, so the windowed context is streamed once per KV head.
// Warp roles: warp 0 issues the TMA loads of 128-key K/V tiles (two-stage pipeline),
// warp 1 issues the tcgen05 MMAs, warps 2-9 run the softmax (two warps per TMEM lane
// quarter, each taking half of the query columns).
//   S^T = K Q^T:  keys are the MMA's M side (128 TMEM lanes, one key per softmax thread);
//                 the N side holds the query rows twice, as the bf16 hi and lo halves of
//                 the fp32 queries, so one MMA gives both products and each thread adds
//                 its two columns.
//   O^T += V^T P^T: d is the M side, the N side holds the probabilities' bf16 hi and lo
//                 halves (written by the softmax threads into shared memory, each key its
//                 own row); the two halves are added once, at the end.
// Keys are taken in ring-slot order (the ring holds rotated keys, so the order of keys
// does not matter to the softmax): a tile is 128 consecutive slots, loaded by one 2-D TMA
// box per 64-column half, and never wraps.  The softmax keeps a reference maximum per
// query and rescales only when a tile exceeds it by more than 2^8 (the probabilities stay
// below 256, well inside bf16); the exact maxima and the row sums are reduced across the
// 128 threads through shared memory.  The block's own 16 keys (hi and lo rows)
// form the last tile of the last split.  Splits write unnormalised partials (O, m, l) and
// merge inside the launch.
#include "bd_device.cuh"
#include "bd_internal.h"
#include "bd_kernels.h"

#include <climits>

namespace bd {

BD_DEFINE_ERROR_TAKER(take_error_word_att)

constexpr int kAttRows = 64;         // query rows per (request, KV head): G*W <= 64
constexpr int kTileKeys = 128;       // context keys per tile (the S MMA's M side)
constexpr int kAttThreads = 320;     // producer warp, MMA warp, eight softmax warps
constexpr int kSoftThreads = 256;
constexpr int kBarSoft = 1;          // named barrier of the softmax warps
constexpr int kBarVote = 2;          // their votes (barrier with an OR reduction)
constexpr int kMaxSplits = 8;        // key splits of one (request, KV head): one portable cluster
constexpr uint32_t kAtom = 16384;    // 128 rows x 128 bytes (64 bf16 of each row)
// shared memory (offsets from the 1024-aligned base); every tile is [2 atoms][128 rows][128 B]
constexpr uint32_t kOffQ = 0;                       // rows 0..63 hi, 64..127 lo queries
constexpr uint32_t kOffK = 2 * kAtom;               // [2 stages] key tiles
constexpr uint32_t kOffV = kOffK + 2 * 2 * kAtom;   // [2 stages] value tiles
constexpr uint32_t kOffP = kOffV + 2 * 2 * kAtom;   // atom 0: hi probabilities, atom 1: lo
constexpr uint32_t kOffRed = kOffP + 2 * kAtom;     // m_ref[64], alpha[64], l[64], q_row[64], red[4][64]
constexpr uint32_t kOffBar = kOffRed + 8 * 64 * 4;
constexpr int kNumBars = 16;  // full_k/v[2], empty_k/v[2], sfull[2], sfree[2], pfull, pvdone, qready, qtma
constexpr size_t kAttSmem = kOffBar + kNumBars * 8 + 16 + 1024;
// TMEM columns: S^T double buffer at 0 and 128, O^T at 256
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;

struct AttMaps {
  CUtensorMap ring_k, ring_v;  // [B*Hkv*cap rows, D], box 128 rows x 64
  CUtensorMap blk_k, blk_v;    // [2*B*Hkv*W rows (hi plane, lo plane), D], box 16 rows x 64
  CUtensorMap q;               // [2*B*W rows (hi plane, lo plane), Hq*D], box W rows x 64
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// 2^x (ex2.approx.ftz: relative error about 2^-22; 2^-inf = 0)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// (x0, x1) -> packed bf16 hi pair and the packed bf16 pair of the residuals x - hi
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  uint32_t hv, lv;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hv) : "f"(x1), "f"(x0));
  const float h0 = __uint_as_float(hv << 16), h1 = __uint_as_float(hv & 0xffff0000u);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lv) : "f"(x1 - h1), "f"(x0 - h0));
  hi = hv;
  lo = lv;
}
// Position of ring slot s of a request at frontier F (the ring holds [F - cap, F) when
// F >= cap, else positions 0..F-1 at their own slots).
__device__ __forceinline__ long long slot_position(long long F, int cap, int s) {
  if (F < cap) return s;
  const long long base = F - cap;
  long long d = (static_cast<long long>(s) - base) % cap;
  if (d < 0) d += cap;
  return base + d;
}

// ------------------------------------------------------------------ producer (one thread)
// K and V tiles have stages of their own: a K stage is free once the S MMA that read it has
// completed, a V stage once its P.V has; both streams are polled without blocking.
template <int D>
__device__ void att_producer(const AttMaps &maps, const AttArgs &a, uint8_t *sm, uint64_t *full_k,
                             uint64_t *full_v, uint64_t *empty_k, uint64_t *empty_v, uint64_t *qtma,
                             int b, int g, long long F, int t_begin, int n_ctx, int nt,
                             volatile int *sabort, int &issued_k, int &issued_v) {
  constexpr int NB = D / 64;  // 64-column boxes per row
  const uint64_t pol_ring = policy_evict_first();
  const uint64_t pol_blk = policy_evict_last();
  const int cap = a.cap;
  const int row0 = (b * a.n_kv_heads + g) * cap;
  const int brow = (b * a.n_kv_heads + g) * a.W;
  const int lo_row = a.B * a.n_kv_heads * a.W;
  // one operand (K: v = 0, V: v = 1) of tile t into its stage t & 1
  auto issue = [&](int t, int v) {
    uint64_t *bar = v ? &full_v[t & 1] : &full_k[t & 1];
    uint8_t *dst = sm + (v ? kOffV : kOffK) + (t & 1) * 2 * kAtom;
    const CUtensorMap *ring = v ? &maps.ring_v : &maps.ring_k;
    const CUtensorMap *blk = v ? &maps.blk_v : &maps.blk_k;
    if (t < n_ctx) {
      const int s0 = (t_begin + t) * kTileKeys;
      mbar_arrive_expect_tx(bar, NB * kAtom);
#pragma unroll
      for (int kb = 0; kb < NB; ++kb) tma_load_2d(dst + kb * kAtom, ring, bar, kb * 64, row0 + s0, pol_ring);
    } else {  // the block's keys/values: hi rows to tile rows 0..15, lo rows to 16..31
      mbar_arrive_expect_tx(bar, 2u * NB * 16 * 128);
#pragma unroll
      for (int kb = 0; kb < NB; ++kb) {
        tma_load_2d(dst + kb * kAtom, blk, bar, kb * 64, brow, pol_blk);
        tma_load_2d(dst + kb * kAtom + 16 * 128, blk, bar, kb * 64, lo_row + brow, pol_blk);
      }
    }
    if (v) issued_v = t + 1; else issued_k = t + 1;
  };
  // The ring holds context written before this round, except the positions >= F - n_guard
  // that this round's catch-up may store (the previous kernel): a first tile without them
  // is fetched before waiting for the previous kernel.
  auto safe = [&](int t) {
    if (t >= n_ctx) return false;
    if (a.n_guard == 0) return true;
    // guard positions [max(0, F - n_guard), F) occupy n consecutive slots from g0 (mod cap)
    const long long p0 = F - a.n_guard > 0 ? F - a.n_guard : 0;
    const int n = static_cast<int>(F - p0);
    if (n >= cap) return false;
    const int g0 = static_cast<int>(p0 % cap);
    const int s0 = (t_begin + t) * kTileKeys, s1 = s0 + kTileKeys;  // the tile's slots [s0, s1)
    const int e0 = g0 + n;                                          // guard slots [g0, e0) and,
    return (e0 <= s0 || g0 >= s1) && (e0 - cap <= s0);             // wrapped, [0, e0 - cap)
  };
  int tk = 0, tv = 0;
  if (nt > 0 && safe(0)) {
    issue(0, 0);
    issue(0, 1);
    tk = tv = 1;
  }
  pdl_wait();
  if (qtma != nullptr) {  // the query tile: hi rows 0..63, lo rows 64..127, W rows per head
    const int G = a.n_q_heads / a.n_kv_heads, W = a.W, T = a.B * a.W;
    mbar_arrive_expect_tx(qtma, static_cast<uint32_t>(2 * G * NB * W * 128));
    for (int p = 0; p < 2; ++p)
      for (int hh = 0; hh < G; ++hh)
#pragma unroll
        for (int kb = 0; kb < NB; ++kb)
          tma_load_2d(sm + kOffQ + kb * kAtom + (p * 64 + hh * W) * 128, &maps.q, qtma,
                      (g * G + hh) * D + kb * 64, p * T + b * W, pol_blk);
  }
  unsigned long long last = globaltimer();
  while (tk < nt || tv < nt) {
    if (*sabort) return;
    bool prog = false;
    if (tk < nt && (tk < 2 || mbar_test_wait(&empty_k[tk & 1], ((tk >> 1) - 1) & 1))) {
      issue(tk++, 0);
      prog = true;
    }
    if (tv < nt && tv < tk && (tv < 2 || mbar_test_wait(&empty_v[tv & 1], ((tv >> 1) - 1) & 1))) {
      issue(tv++, 1);
      prog = true;
    }
    if (prog) {
      last = globaltimer();
    } else if (globaltimer() - last > kWaitLimitNs) {
      atomicOr(&g_error_word, DEVERR_TIMEOUT);
      *sabort = 1;
      return;
    }
  }
}

// ------------------------------------------------------------------ MMA issuer (one thread)
template <int D>
__device__ void att_mma(uint8_t *sm, uint64_t *full_k, uint64_t *full_v, uint64_t *empty_k,
                        uint64_t *empty_v, uint64_t *sfull, uint64_t *sfree, uint64_t *pfull,
                        uint64_t *pvdone, uint64_t *qready, uint64_t *qtma, uint32_t tmem, int n_ctx,
                        int nt, volatile int *sabort) {
  const uint32_t idesc_s = umma_idesc(1, 128, 128);                           // both K-major
  const uint32_t idesc_o = umma_idesc(1, 128, 128) | (1u << 15) | (1u << 16);  // both MN-major
  if (!mbar_wait(qready, 0) || (qtma != nullptr && !mbar_wait(qtma, 0))) {
    *sabort = 1;
    return;
  }
  tc_fence_after();
  const uint32_t q_base = smem_u32(sm + kOffQ);
  const uint32_t p_base = smem_u32(sm + kOffP);
  // S of tile ns needs its K tile and a free S buffer; P.V of tile np needs its
  // probabilities.  Both are polled without blocking, so a P.V is issued as soon as its
  // probabilities are ready (the stage it frees is what the producer refills next).
  int ns = 0, np = 0;
  unsigned long long last = globaltimer();
  while (np < nt) {
    if (*sabort) return;
    bool prog = false;
    if (ns < nt && mbar_test_wait(&full_k[ns & 1], (ns >> 1) & 1) &&
        (ns < 2 || mbar_test_wait(&sfree[ns & 1], ((ns >> 1) - 1) & 1))) {
      tc_fence_after();
      const uint32_t k_base = smem_u32(sm + kOffK + (ns & 1) * 2 * kAtom);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kAtom + (kk & 3) * 32;
        umma_bf16(tmem + (ns & 1) * 128, umma_desc_sw128(k_base + off), umma_desc_sw128(q_base + off),
                  idesc_s, kk > 0 ? 1u : 0u);
      }
      umma_commit(&sfull[ns & 1]);
      umma_commit(&empty_k[ns & 1]);  // the K stage is free
      ++ns;
      prog = true;
    }
    if (np < ns && mbar_test_wait(pfull, np & 1) && mbar_test_wait(&full_v[np & 1], (np >> 1) & 1)) {
      tc_fence_after();
      const uint32_t v_base = smem_u32(sm + kOffV + (np & 1) * 2 * kAtom);
      const int nk = np < n_ctx ? kTileKeys / 16 : 2;  // the block tile has 32 key rows
      for (int kk = 0; kk < nk; ++kk)
        umma_bf16(tmem + kTmemO, umma_desc_sw128_mn(v_base + kk * 2048, kAtom, 1024),
                  umma_desc_sw128_mn(p_base + kk * 2048, kAtom, 1024), idesc_o,
                  (np > 0 || kk > 0) ? 1u : 0u);
      umma_commit(&empty_v[np & 1]);  // the V stage is free
      umma_commit(pvdone);            // the probabilities are consumed, O^T is up to date
      ++np;
      prog = true;
    }
    if (prog) {
      last = globaltimer();
    } else if (globaltimer() - last > kWaitLimitNs) {
      atomicOr(&g_error_word, DEVERR_TIMEOUT);
      *sabort = 1;
      return;
    }
  }
}

// Columns [c, c+32) and [c+64, c+96) of this thread's TMEM lane (taddr = lane base + c),
// added: the hi and lo halves of one product.
__device__ __forceinline__ void tmem_pair32(uint32_t taddr, float (&v)[32]) {
  uint32_t hv[32], lv[32];
  tmem_ld32_nowait(taddr, hv);
  tmem_ld32_nowait(taddr + 64, lv);
  tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(hv[j]) + __uint_as_float(lv[j]);
}

// Butterfly reduce-scatter of 32 values over the warp: afterwards v[0] of lane j holds the
// warp-wide sum of entry j.  At each step a lane keeps one half of its entries and adds its
// partner's copy of that half.
template <int N, int O>
__device__ __forceinline__ void bfly_sum_step(float (&v)[32], int lane) {
  const bool up = (lane & O) != 0;
#pragma unroll
  for (int j = 0; j < N / 2; ++j) {
    const float send = up ? v[j] : v[j + N / 2];
    const float keep = up ? v[j + N / 2] : v[j];
    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, O);
  }
}
__device__ __forceinline__ void bfly_sum32(float (&v)[32], int lane) {
  bfly_sum_step<32, 16>(v, lane);
  bfly_sum_step<16, 8>(v, lane);
  bfly_sum_step<8, 4>(v, lane);
  bfly_sum_step<4, 2>(v, lane);
  bfly_sum_step<2, 1>(v, lane);
}

// Final outputs of one thread (output dim kr, queries h*32 .. h*32+31) from unnormalised
// sums o and row sums l, token-major [B*W][Hq*D]: one fp16 plane (out_f16, the operand of
// an fp16 output projection) or bf16 hi (and lo) planes.
__device__ __forceinline__ void write_out(const AttArgs &a, int b, int g, int kr, int h,
                                          const float *l, const float (&o)[32]) {
  const int D = a.head_dim, W = a.W, G = a.n_q_heads / a.n_kv_heads, R = G * W;
  if (kr >= D) return;
  bool bad = false;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int q = h * 32 + j;
    if (q < R) {
      const int hh = q / W, i = q - hh * W;
      const float L = l[q];
      const float y = L > 0.f ? o[j] / L : 0.f;
      const size_t idx = (static_cast<size_t>(b) * W + i) * a.n_q_heads * D +
                         static_cast<size_t>(g * G + hh) * D + kr;
      if (a.out_f16) {
        bad |= f16_out_of_range(y);
        static_cast<__half *>(a.out)[idx] = __float2half_rn(y);
      } else {
        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out);
        const __nv_bfloat16 hv = __float2bfloat16_rn(y);
        out[idx] = hv;
        if (a.out_lo) out[a.out_lo + idx] = __float2bfloat16_rn(y - __bfloat162float(hv));
      }
    }
  }
  flag_f16_range(bad);
}

// Merge of the cluster's partials (O, m, l) for query rows r0 .. r1-1 of (request b, KV
// head g), by the 256 softmax threads of one CTA:
//   out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s,  M = max over splits with l_s > 0,
// reading split s's partial from CTA s of the cluster (distributed shared memory): its
// [query][D] fp32 tile at kOffP and its per-query m, l.  Each thread takes 4 output columns
// of a row per chunk and NCH chunks at a time, and issues every remote load they need (the
// rows' m and l of the SM <= kMaxSplits splits and up to four splits' columns) before any
// arithmetic, so NCH chunks cost one remote round trip (plus one per further group of four
// splits) and need no barrier; splits are added in rank order.
template <int D, int NCH, int SM>
__device__ void merge_cluster(const AttArgs &a, int b, int g, int r0, int r1, int tid, uint8_t *sm) {
  constexpr int C4 = D / 4;             // float4 chunks per row
  constexpr int SB = SM < 4 ? SM : 4;   // splits whose columns are loaded up front
  const int S = a.n_splits, total = (r1 - r0) * C4;
  const int G = a.n_q_heads / a.n_kv_heads;
  const uint32_t ml_base = smem_u32(sm + kOffRed);  // m_ref[64], then alpha[64], l[64]
  const uint32_t p_base = smem_u32(sm + kOffP);
  __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out);
  for (int c0 = tid; c0 < total; c0 += NCH * kSoftThreads) {
    float m[NCH][SM], l[NCH][SM];
    float4 v[NCH][SB];
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
      const int c = c0 + k * kSoftThreads;
      if (c >= total) break;
      const int r = c / C4, q = r0 + r;
      const uint32_t o_off = p_base + static_cast<uint32_t>((q * D + 4 * (c - r * C4)) * 4);
#pragma unroll
      for (int sp = 0; sp < SM; ++sp)
        if (sp < S) {
          const uint32_t rm = cluster_map(ml_base, static_cast<uint32_t>(sp));
          m[k][sp] = ld_cluster_f32(rm + q * 4);
          l[k][sp] = ld_cluster_f32(rm + (128 + q) * 4);
          if (sp < SB) v[k][sp] = ld_cluster_f4(cluster_map(o_off, static_cast<uint32_t>(sp)));
        }
    }
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
      const int c = c0 + k * kSoftThreads;
      if (c >= total) break;
      const int r = c / C4, d4 = c - r * C4, q = r0 + r;
      const uint32_t o_off = p_base + static_cast<uint32_t>((q * D + 4 * d4) * 4);
      float M = -INFINITY;
#pragma unroll
      for (int sp = 0; sp < SM; ++sp)
        if (sp < S && l[k][sp] > 0.f) M = fmaxf(M, m[k][sp]);
      float L = 0.f;
      float w[SM];
#pragma unroll
      for (int sp = 0; sp < SM; ++sp)
        if (sp < S) {
          w[sp] = l[k][sp] > 0.f ? exp2f(m[k][sp] - M) : 0.f;  // the split's weight
          L += w[sp] * l[k][sp];
        }
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int s0 = 0; s0 < SM; s0 += 4) {
        if (s0 >= S) break;
        float4 u[SB];
#pragma unroll
        for (int j = 0; j < SB; ++j)
          if (s0 + j < S)
            u[j] = s0 == 0 ? v[k][j] : ld_cluster_f4(cluster_map(o_off, static_cast<uint32_t>(s0 + j)));
#pragma unroll
        for (int j = 0; j < SB; ++j)
          if (s0 + j < S) {
            const float ws = w[s0 + j];
            acc.x += ws * u[j].x;
            acc.y += ws * u[j].y;
            acc.z += ws * u[j].z;
            acc.w += ws * u[j].w;
          }
      }
      const float il = L > 0.f ? 1.f / L : 0.f;
      const int hh = q / a.W, i = q - hh * a.W;
      const size_t idx = (static_cast<size_t>(b) * a.W + i) * a.n_q_heads * D +
                         static_cast<size_t>(g * G + hh) * D + 4 * d4;
      const float y0 = acc.x * il, y1 = acc.y * il, y2 = acc.z * il, y3 = acc.w * il;
      if (a.out_f16) {
        flag_f16_range(f16_out_of_range(y0) || f16_out_of_range(y1) || f16_out_of_range(y2) ||
                       f16_out_of_range(y3));
        const __half2 h01 = __floats2half2_rn(y0, y1), h23 = __floats2half2_rn(y2, y3);
        *reinterpret_cast<uint2 *>(static_cast<__half *>(a.out) + idx) =
            make_uint2(*reinterpret_cast<const uint32_t *>(&h01), *reinterpret_cast<const uint32_t *>(&h23));
      } else {
        uint32_t hw[2], lw[2];
        split_bf16x2(y0, y1, hw[0], lw[0]);
        split_bf16x2(y2, y3, hw[1], lw[1]);
        *reinterpret_cast<uint2 *>(out + idx) = make_uint2(hw[0], hw[1]);
        if (a.out_lo) *reinterpret_cast<uint2 *>(out + a.out_lo + idx) = make_uint2(lw[0], lw[1]);
      }
    }
  }
}

// ------------------------------------------------------------------ kernel
template <int D>
__global__ void __launch_bounds__(kAttThreads, 1)
    attention_tc_kernel(const __grid_constant__ AttMaps maps, const __grid_constant__ AttArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float *m_ref_s = reinterpret_cast<float *>(sm + kOffRed);  // per query: reference max (log2 units)
  float *alpha = m_ref_s + 64, *l_fin = alpha + 64;          // rescale factors, row sums
  int *q_row = reinterpret_cast<int *>(l_fin + 64);           // block row of each query
  float *red_max = reinterpret_cast<float *>(q_row + 64);     // [4 warps][64 queries] scratch
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
  uint64_t *full_k = bars, *full_v = bars + 2, *empty_k = bars + 4, *empty_v = bars + 6;
  uint64_t *sfull = bars + 8, *sfree = bars + 10;
  uint64_t *pfull = bars + 12, *pvdone = bars + 13, *qready = bars + 14, *qtma = bars + 15;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNumBars);
  volatile int *sabort = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.n_q_heads / a.n_kv_heads, W = a.W, R = G * W;
  // the frontier is an input of the round, readable before the dependency wait
  const long long F = a.frontier[b];
  const int cap = a.cap;
  const int n_slots = F < cap ? static_cast<int>(F > 0 ? F : 0) : cap;
  const int n_tiles = (n_slots + kTileKeys - 1) / kTileKeys;
  const int per = (n_tiles + a.n_splits - 1) / a.n_splits;
  const int t_begin = min(n_tiles, split * per);
  const int n_ctx = min(n_tiles, t_begin + per) - t_begin;
  const bool do_block = split == a.n_splits - 1;
  const bool q_tma = W % 8 == 0;  // the query tile by TMA (see the softmax warps' Q load)
  const int nt = n_ctx + (do_block ? 1 : 0);

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full_k[i], 1);
      mbar_init(&full_v[i], 1);
      mbar_init(&empty_k[i], 1);
      mbar_init(&empty_v[i], 1);
    }
    mbar_init(&sfull[0], 1);
    mbar_init(&sfull[1], 1);
    mbar_init(&sfree[0], kSoftThreads);
    mbar_init(&sfree[1], kSoftThreads);
    mbar_init(pfull, kSoftThreads);
    mbar_init(pvdone, 1);
    mbar_init(qready, kSoftThreads);
    mbar_init(qtma, 1);
    *sabort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.ring_k);
    tma_prefetch_desc(&maps.ring_v);
    tma_prefetch_desc(&maps.blk_k);
    tma_prefetch_desc(&maps.blk_v);
    tma_prefetch_desc(&maps.q);
  }
  if (warp == 1) {  // TMEM before the trigger: a dependent kernel cannot take it first
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();

  int issued_k = 0, issued_v = 0;
  if (warp == 0) {
    if (lane == 0)
      att_producer<D>(maps, a, sm, full_k, full_v, empty_k, empty_v, q_tma ? qtma : nullptr, b, g, F,
                      t_begin, n_ctx, nt, sabort, issued_k, issued_v);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0)
      att_mma<D>(sm, full_k, full_v, empty_k, empty_v, sfull, sfree, pfull, pvdone, qready,
                 q_tma ? qtma : nullptr, tmem, n_ctx, nt, sabort);
    __syncwarp();
  } else {
    // softmax warps 2..9: lane quarter qd of the tiles (key row / output dim kr), query
    // half h (queries h*32 .. h*32+31)
    const int qd = warp & 3;
    const int kr = qd * 32 + lane;
    const int h = (warp - 2) >> 2;
    const int st_id = tid - 64;  // 0..255 among the softmax threads
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    // every wait is made warp-uniform (the TMEM loads after it are warp-collective); after a
    // wait gives up the others return at once, so all threads still pass the same barriers
    auto wait_ok = [&](uint64_t *bar, uint32_t parity) {
      bool ok = !*sabort && mbar_wait(bar, parity);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) *sabort = 1;
      return ok;
    };
    pdl_wait();
    // query tile (queried rows already scaled by log2(e)/sqrt(D), so the scores come out in
    // log2 units): tile row r (hi plane) and row 64 + r (lo plane) hold query r =
    // head_in_group*W + i.  With W a multiple of 8 the producer loads it by TMA (each
    // head's W rows land 1024-byte aligned) and these threads only clear the rows past R;
    // else each thread copies one 64-column half of one plane row.
    {
      const int n = st_id & 127, half = st_id >> 7, plane = n >> 6, r = n & 63;
      if (q_tma) {
        if (half * 64 < D && r >= R)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4 *>(sm + kOffQ + half * kAtom + n * 128 + (c << 4)) = make_uint4(0, 0, 0, 0);
      } else if (half * 64 < D) {
        const bool ok = r < R;
        const int hh = ok ? r / W : 0, i = ok ? r % W : 0;
        const uint4 *src = reinterpret_cast<const uint4 *>(
            static_cast<const __nv_bfloat16 *>(a.q) + (plane ? a.q_lo : 0) +
            (static_cast<size_t>(b) * W + i) * a.n_q_heads * D + static_cast<size_t>(g * G + hh) * D +
            half * 64);
        uint4 v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) v[c] = ok ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4 *>(sm + kOffQ + half * kAtom + n * 128 + ((c ^ (n & 7)) << 4)) = v[c];
      }
    }
    if (st_id < 64) {
      const int q = st_id;
      q_row[q] = q < R ? q % W : (1 << 20);  // block row of query q (never visible past R)
      m_ref_s[q] = -1e30f;
    }
    fence_proxy_async_shared();
    mbar_arrive(qready);
    named_bar(kBarSoft, kSoftThreads);

    // reference maxima (log2 units) of this thread's 32 queries; a finite start value, so
    // that a hidden key (-inf) gives a zero probability before the first reference is set
    constexpr float kNoRef = -1e30f;
    float mr[32], lsum[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      mr[j] = kNoRef;
      lsum[j] = 0.f;
    }
    uint8_t *prow = sm + kOffP + kr * 128;
    const uint32_t swz = static_cast<uint32_t>(kr & 7);
    // ring slot of position F - cap (the oldest) once the ring is full
    const int base_slot = F >= cap ? static_cast<int>(F % cap) : 0;
    for (int t = 0; t < nt; ++t) {
      const int sb = t & 1;
      float s[32];
      if (wait_ok(&sfull[sb], (t >> 1) & 1)) {
        tc_fence_after();
        tmem_pair32(tmem + lane_off + sb * 128 + h * 32, s);
      }
      tc_fence_before();
      mbar_arrive(&sfree[sb]);  // the S buffer may take the tile after next
      // hide the keys a query's block row may not see (-inf)
      if (t < n_ctx) {
        const int slot = (t_begin + t) * kTileKeys + kr;
        int vis_rows;  // this key is seen by block rows 0 .. vis_rows-1
        if (slot >= n_slots) {
          vis_rows = 0;
        } else if (a.window <= 0) {
          vis_rows = W;
        } else {  // position p sits in the window of row i iff p >= F + i - window + 1
          int d = slot - base_slot;
          if (d < 0) d += cap;
          const int m = F >= cap ? d + a.window - 1 - cap : slot - static_cast<int>(F) + a.window - 1;
          vis_rows = m < 0 ? 0 : (m >= W ? W : m + 1);
        }
        if (vis_rows == 0) {
#pragma unroll
          for (int j = 0; j < 32; ++j) s[j] = -INFINITY;
        } else if (vis_rows < W) {
#pragma unroll
          for (int j = 0; j < 32; ++j) s[j] = q_row[h * 32 + j] < vis_rows ? s[j] : -INFINITY;
        }
      } else {  // the block tile: lanes 16..31 of quarter 0 hold the lo key rows
        if (qd == 0) {
#pragma unroll
          for (int j = 0; j < 32; ++j) s[j] += __shfl_down_sync(0xffffffffu, s[j], 16);
        }
        const bool key_ok = qd == 0 && kr < W;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int i = q_row[h * 32 + j];
          const bool vis = key_ok && i < W && (!a.causal || kr <= i) &&
                           (a.window <= 0 || abs(kr - i) < a.window);
          s[j] = vis ? s[j] : -INFINITY;
        }
      }
      // the reference moves when a tile exceeds it by more than 2^8 (s stays the raw score:
      // before the first reference s - m_ref would lose s against the start value)
      float dmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < 32; ++j) dmax = fmaxf(dmax, s[j] - mr[j]);
      const bool need = named_bar_or(kBarVote, kSoftThreads, dmax > 8.f);
      if (need) {  // new reference maxima (exact over this tile): rescale l and O^T
        // column maxima: warp reduction on order-preserving integer images, then the
        // four warps of this query half through shared memory
        int mine = 0;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          int bits = __float_as_int(s[j]);
          bits = bits >= 0 ? bits : bits ^ 0x7FFFFFFF;
          const int wmax = __reduce_max_sync(0xffffffffu, bits);
          mine = lane == j ? wmax : mine;
        }
        mine = mine >= 0 ? mine : mine ^ 0x7FFFFFFF;
        red_max[qd * 64 + h * 32 + lane] = __int_as_float(mine);
        if (t > 0) wait_ok(pvdone, (t - 1) & 1);  // O^T stable before it is rescaled
        named_bar(kBarSoft, kSoftThreads);
        if (st_id < 64) {
          const float tm = fmaxf(fmaxf(red_max[st_id], red_max[64 + st_id]),
                                 fmaxf(red_max[128 + st_id], red_max[192 + st_id]));
          const float m_old = m_ref_s[st_id], m_new = fmaxf(m_old, tm);
          alpha[st_id] = exp2f(m_old - m_new);
          m_ref_s[st_id] = m_new;
        }
        named_bar(kBarSoft, kSoftThreads);
        const float *arow = alpha + h * 32;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          mr[j] = m_ref_s[h * 32 + j];
          lsum[j] *= arow[j];
        }
        if (t > 0 && __all_sync(0xffffffffu, *sabort == 0)) {  // O^T row kr, this half's columns
          tc_fence_after();
#pragma unroll 1
          for (int part = 0; part < 2; ++part) {  // hi columns, then lo columns
            const uint32_t ta = tmem + lane_off + kTmemO + part * 64 + h * 32;
            uint32_t o[32];
            tmem_ld32_nowait(ta, o);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * arow[j]);
            tmem_st32(ta, o);
          }
          tmem_st_wait();
        }
      } else if (t > 0) {
        wait_ok(pvdone, (t - 1) & 1);  // the previous tile's P.V has read the P tile
      }
      // probabilities, bf16 hi and lo halves, key row kr of the P^T tile
      const bool dup = t >= n_ctx && qd == 0 && kr >= 16;  // block lo-key rows repeat 0..15
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t ph[4], pl[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = c * 8 + 2 * e;
          const float p0 = ex2_approx(s[j] - mr[j]), p1 = ex2_approx(s[j + 1] - mr[j + 1]);
          lsum[j] += p0;
          lsum[j + 1] += p1;
          split_bf16x2(p0, p1, ph[e], pl[e]);
        }
        if (!dup) {
          const uint32_t off = static_cast<uint32_t>(((h * 4 + c) ^ swz) << 4);
          *reinterpret_cast<uint4 *>(prow + off) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
          *reinterpret_cast<uint4 *>(prow + kAtom + off) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
        }
      }
      if (t >= n_ctx && qd == 0) {
        __syncwarp();
        if (dup) {  // kr & 7 == (kr - 16) & 7: the same swizzle positions
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint32_t off = static_cast<uint32_t>(((h * 4 + c) ^ swz) << 4);
            *reinterpret_cast<uint4 *>(prow + off) = *reinterpret_cast<const uint4 *>(prow - 16 * 128 + off);
            *reinterpret_cast<uint4 *>(prow + kAtom + off) =
                *reinterpret_cast<const uint4 *>(prow - 16 * 128 + kAtom + off);
          }
        }
      }
      fence_proxy_async_shared();
      tc_fence_before();
      mbar_arrive(pfull);
    }
    if (nt > 0) wait_ok(pvdone, (nt - 1) & 1);
    const bool abort = named_bar_or(kBarVote, kSoftThreads, *sabort != 0);
    if (!abort) {
      // row sums: butterfly over the warp (lane j ends with query h*32 + j), then the four
      // warps of this query half
      bfly_sum32(lsum, lane);
      red_max[qd * 64 + h * 32 + lane] = lsum[0];
      named_bar(kBarSoft, kSoftThreads);
      if (st_id < 64)
        l_fin[st_id] = (red_max[st_id] + red_max[64 + st_id]) + (red_max[128 + st_id] + red_max[192 + st_id]);
      named_bar(kBarSoft, kSoftThreads);
      // O^T row kr (output dim d = kr): query q sits in columns q and q + 64
      float o[32];
      if (nt > 0) {
        tc_fence_after();
        tmem_pair32(tmem + lane_off + kTmemO + h * 32, o);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = 0.f;
      }
      if (a.n_splits == 1) {
        write_out(a, b, g, kr, h, l_fin, o);
      } else if (kr < D) {  // this split's partial, for the cluster's merge: [query][D] fp32
        float *po = reinterpret_cast<float *>(sm + kOffP);
#pragma unroll
        for (int j = 0; j < 32; ++j) po[(h * 32 + j) * D + kr] = o[j];
      }
    }
  }
  if (a.n_splits > 1) {
    // the splits of (b, g) form one cluster: merge their partials through distributed
    // shared memory (every thread of every CTA passes both cluster barriers)
    cluster_sync();
    if (warp >= 2) {
      const int rp = (R + a.n_splits - 1) / a.n_splits;
      const int r0 = min(R, split * rp), r1 = min(R, (split + 1) * rp);
      // more chunks in flight when fewer splits' values are loaded per chunk
      if (a.n_splits <= 2)
        merge_cluster<D, 4, 2>(a, b, g, r0, r1, tid - 64, sm);
      else if (a.n_splits <= 4)
        merge_cluster<D, 2, 4>(a, b, g, r0, r1, tid - 64, sm);
      else
        merge_cluster<D, 1, kMaxSplits>(a, b, g, r0, r1, tid - 64, sm);
    }
    cluster_sync();  // no CTA leaves while the others still read its partial
  }
  tc_fence_before();
  __syncthreads();
  if (*sabort && warp == 0 && lane == 0) {
    // a wait gave up: let the loads still in flight land before the CTA exits (bounded)
    for (int t = max(0, issued_k - 2); t < issued_k; ++t) mbar_wait(&full_k[t & 1], (t >> 1) & 1);
    for (int t = max(0, issued_v - 2); t < issued_v; ++t) mbar_wait(&full_v[t & 1], (t >> 1) & 1);
    if (q_tma) mbar_wait(qtma, 0);
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ fp32 path
// Context keys [p_lo, F) of request b: the window's oldest visible position, clipped to
// the ring's live interval [F - cap, F).
struct AttGeom {
  long long F;
  int p_lo, n_ctx;
};
__device__ __forceinline__ AttGeom att_geom(const AttArgs &a, int b) {
  AttGeom g;
  g.F = a.frontier[b];
  long long lo = a.window > 0 ? g.F - a.window + 1 : 0;
  if (g.F - a.cap > lo) lo = g.F - a.cap;
  if (lo < 0) lo = 0;
  g.p_lo = static_cast<int>(lo);
  g.n_ctx = g.F > lo ? static_cast<int>(g.F - lo) : 0;
  return g;
}
// Is context key k (0-based from p_lo) visible from block row i?
__device__ __forceinline__ bool ctx_visible(const AttArgs &a, const AttGeom &g, int i, int k) {
  if (k >= g.n_ctx) return false;
  const long long p = g.p_lo + k;
  return a.window <= 0 || (g.F + i) - p < a.window;
}
// Is block key j visible from block row i?
__device__ __forceinline__ bool blk_visible(const AttArgs &a, int i, int j) {
  if (j >= a.W) return false;
  if (a.window > 0 && abs(j - i) >= a.window) return false;
  return !a.causal || j <= i;
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
  const AttGeom g = att_geom(a, b);
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

int attention_rows_max() { return kAttRows; }
int attention_tile_keys() { return kTileKeys; }
int attention_max_splits() { return kMaxSplits; }

template <int D>
static cudaError_t launch_tc(const AttMaps &m, const AttArgs &a, cudaStream_t stream) {
  static bool set = false;  // one flag per head dimension
  if (!set) {
    const cudaError_t e = cudaFuncSetAttribute(attention_tc_kernel<D>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(kAttSmem));
    if (e != cudaSuccess) return e;
    set = true;
  }
  return launch_pdl_cluster(attention_tc_kernel<D>, dim3(a.n_splits, a.n_kv_heads, a.B),
                            dim3(kAttThreads), kAttSmem, stream, a.n_splits, m, a);
}

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
  // bf16: the query and block planes must be contiguous (lo plane right after hi)
  const int D = a.head_dim;
  const long long T = static_cast<long long>(a.B) * a.W;
  if (a.q_lo != static_cast<size_t>(T * a.n_q_heads * D) ||
      a.blk_lo != static_cast<size_t>(T * a.n_kv_heads * D))
    return "attention: hi/lo planes of the queries and block keys must be contiguous";
  AttMaps m;
  const int ring_rows = a.B * a.n_kv_heads * a.cap;
  const int blk_rows = 2 * a.B * a.n_kv_heads * a.W;
  std::string err;
  if (!(err = make_tensor_map_2d(&m.ring_k, a.ring_k, GT_BF16, D, ring_rows, 64, kTileKeys, true)).empty() ||
      !(err = make_tensor_map_2d(&m.ring_v, a.ring_v, GT_BF16, D, ring_rows, 64, kTileKeys, true)).empty() ||
      !(err = make_tensor_map_2d(&m.blk_k, a.blk_k, GT_BF16, D, blk_rows, 64, 16, true)).empty() ||
      !(err = make_tensor_map_2d(&m.blk_v, a.blk_v, GT_BF16, D, blk_rows, 64, 16, true)).empty() ||
      !(err = make_tensor_map_2d(&m.q, a.q, GT_BF16, a.n_q_heads * D, static_cast<int>(2 * T), 64,
                                 a.W <= 256 ? a.W : 256, true)).empty())
    return err;
  e = D == 128 ? launch_tc<128>(m, a, stream) : launch_tc<64>(m, a, stream);
  if (e != cudaSuccess) return std::string("attention launch: ") + cudaGetErrorString(e);
  return {};
}

}  // namespace bd
