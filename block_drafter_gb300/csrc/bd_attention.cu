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
// warp 1 issues the tcgen05 MMAs, warps 2-5 (one TMEM lane quarter each) run the softmax.
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
constexpr int kAttThreads = 192;     // producer warp, MMA warp, four softmax warps
constexpr int kSoftThreads = 128;
constexpr int kBarSoft = 1;          // named barrier of the softmax warps
constexpr int kBarVote = 2;          // their votes (barrier with an OR reduction)
constexpr uint32_t kAtom = 16384;    // 128 rows x 128 bytes (64 bf16 of each row)
// shared memory (offsets from the 1024-aligned base); every tile is [2 atoms][128 rows][128 B]
constexpr uint32_t kOffQ = 0;                       // rows 0..63 hi, 64..127 lo queries
constexpr uint32_t kOffK = 2 * kAtom;               // [2 stages] key tiles
constexpr uint32_t kOffV = kOffK + 2 * 2 * kAtom;   // [2 stages] value tiles
constexpr uint32_t kOffP = kOffV + 2 * 2 * kAtom;   // atom 0: hi probabilities, atom 1: lo
constexpr uint32_t kOffRed = kOffP + 2 * kAtom;     // float m_ref[64], alpha[64], l[64]
constexpr uint32_t kOffBar = kOffRed + 3 * 64 * 4;
constexpr int kNumBars = 11;  // full[2], empty[2], sfull[2], sfree[2], pfull, pvdone, qready
constexpr size_t kAttSmem = kOffBar + kNumBars * 8 + 16 + 1024;
// TMEM columns: S^T double buffer at 0 and 128, O^T at 256
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;

struct AttMaps {
  CUtensorMap ring_k, ring_v;  // [B*Hkv*cap rows, D], box 128 rows x 64
  CUtensorMap blk_k, blk_v;    // [2*B*Hkv*W rows (hi plane, lo plane), D], box 16 rows x 64
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// Column reduction of a [128 threads][64] value table through shared memory (the free
// probability tile): element (row r, column q) sits at r*64 + (q ^ (r & 31)), so both the
// row writes of a warp and the column reads of 32 threads touch 32 distinct banks.
__device__ __forceinline__ void table_store(float *scr, int r, const float (&v)[64]) {
#pragma unroll
  for (int q = 0; q < 64; ++q) scr[r * 64 + (q ^ (r & 31))] = v[q];
}
template <bool MAX>
__device__ __forceinline__ float table_column(const float *scr, int q) {
  float acc = MAX ? -INFINITY : 0.f;
#pragma unroll 8
  for (int r = 0; r < 128; ++r) {
    const float x = scr[r * 64 + (q ^ (r & 31))];
    acc = MAX ? fmaxf(acc, x) : acc + x;
  }
  return acc;
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
      named_bar(kBarSoft, kSoftThreads);
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
template <int D>
__device__ void att_producer(const AttMaps &maps, const AttArgs &a, uint8_t *sm, uint64_t *full,
                             uint64_t *empty, int b, int g, long long F, int t_begin, int n_ctx,
                             int nt, volatile int *sabort, int &issued) {
  constexpr int NB = D / 64;  // 64-column boxes per row
  const uint64_t pol_ring = policy_evict_first();
  const int cap = a.cap;
  const int row0 = (b * a.n_kv_heads + g) * cap;
  auto issue = [&](int t) {
    const int st = t & 1;
    uint64_t *bar = &full[st];
    uint8_t *dk = sm + kOffK + st * 2 * kAtom;
    uint8_t *dv = sm + kOffV + st * 2 * kAtom;
    if (t < n_ctx) {
      const int s0 = (t_begin + t) * kTileKeys;
      mbar_arrive_expect_tx(bar, 2u * NB * kAtom);
#pragma unroll
      for (int kb = 0; kb < NB; ++kb) {
        tma_load_2d(dk + kb * kAtom, &maps.ring_k, bar, kb * 64, row0 + s0, pol_ring);
        tma_load_2d(dv + kb * kAtom, &maps.ring_v, bar, kb * 64, row0 + s0, pol_ring);
      }
    } else {  // the block's keys/values: hi rows to tile rows 0..15, lo rows to 16..31
      const int brow = (b * a.n_kv_heads + g) * a.W;
      const int lo_row = a.B * a.n_kv_heads * a.W;
      const uint64_t pol = policy_evict_last();
      mbar_arrive_expect_tx(bar, 4u * NB * 16 * 128);
#pragma unroll
      for (int kb = 0; kb < NB; ++kb) {
        tma_load_2d(dk + kb * kAtom, &maps.blk_k, bar, kb * 64, brow, pol);
        tma_load_2d(dk + kb * kAtom + 16 * 128, &maps.blk_k, bar, kb * 64, lo_row + brow, pol);
        tma_load_2d(dv + kb * kAtom, &maps.blk_v, bar, kb * 64, brow, pol);
        tma_load_2d(dv + kb * kAtom + 16 * 128, &maps.blk_v, bar, kb * 64, lo_row + brow, pol);
      }
    }
    issued = t + 1;
  };
  // The ring holds context written before this round, except the positions >= F - n_guard
  // that this round's catch-up may store (the previous kernel): a first tile without them
  // is fetched before waiting for the previous kernel.
  auto safe = [&](int t) {
    if (t >= n_ctx) return false;
    const int s0 = (t_begin + t) * kTileKeys;
    for (int j = 0; j < a.n_guard; ++j) {
      const long long p = F - 1 - j;
      if (p < 0) break;
      const int slot = static_cast<int>(p % cap);
      if (slot >= s0 && slot < s0 + kTileKeys) return false;
    }
    return true;
  };
  int t = 0;
  if (nt > 0 && safe(0)) issue(t++);
  pdl_wait();
  for (; t < nt; ++t) {
    if (t >= 2 && (*sabort || !mbar_wait(&empty[t & 1], ((t >> 1) - 1) & 1))) {
      *sabort = 1;
      return;
    }
    issue(t);
  }
}

// ------------------------------------------------------------------ MMA issuer (one thread)
template <int D>
__device__ void att_mma(uint8_t *sm, uint64_t *full, uint64_t *empty, uint64_t *sfull,
                        uint64_t *sfree, uint64_t *pfull, uint64_t *pvdone, uint64_t *qready,
                        uint32_t tmem, int n_ctx, int nt, volatile int *sabort) {
  const uint32_t idesc_s = umma_idesc(1, 128, 128);                           // both K-major
  const uint32_t idesc_o = umma_idesc(1, 128, 128) | (1u << 15) | (1u << 16);  // both MN-major
  if (!mbar_wait(qready, 0)) {
    *sabort = 1;
    return;
  }
  tc_fence_after();
  const uint32_t q_base = smem_u32(sm + kOffQ);
  const uint32_t p_base = smem_u32(sm + kOffP);
  auto pv = [&](int u) -> bool {
    if (*sabort || !mbar_wait(pfull, u & 1)) return false;
    tc_fence_after();
    const uint32_t v_base = smem_u32(sm + kOffV + (u & 1) * 2 * kAtom);
    const int nk = u < n_ctx ? kTileKeys / 16 : 2;  // the block tile has 32 key rows
    for (int kk = 0; kk < nk; ++kk)
      umma_bf16(tmem + kTmemO, umma_desc_sw128_mn(v_base + kk * 2048, kAtom, 1024),
                umma_desc_sw128_mn(p_base + kk * 2048, kAtom, 1024), idesc_o,
                (u > 0 || kk > 0) ? 1u : 0u);
    umma_commit(&empty[u & 1]);  // the K/V stage is free
    umma_commit(pvdone);         // the probabilities are consumed, O^T is up to date
    return true;
  };
  for (int t = 0; t < nt; ++t) {
    const int st = t & 1;
    if (*sabort || !mbar_wait(&full[st], (t >> 1) & 1) ||
        (t >= 2 && !mbar_wait(&sfree[st], ((t >> 1) - 1) & 1))) {
      *sabort = 1;
      return;
    }
    tc_fence_after();
    const uint32_t k_base = smem_u32(sm + kOffK + st * 2 * kAtom);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (kk >> 2) * kAtom + (kk & 3) * 32;
      umma_bf16(tmem + st * 128, umma_desc_sw128(k_base + off), umma_desc_sw128(q_base + off),
                idesc_s, kk > 0 ? 1u : 0u);
    }
    umma_commit(&sfull[st]);
    if (t >= 1 && !pv(t - 1)) {  // the previous tile's P.V, behind this tile's scores
      *sabort = 1;
      return;
    }
  }
  if (nt > 0 && !pv(nt - 1)) *sabort = 1;
}

// Loads columns [c0, c0+32) and [c0+64, c0+96) of this thread's TMEM lane and returns
// their sums (the hi and lo halves of one product) in v[j0 .. j0+31].
template <int J0>
__device__ __forceinline__ void tmem_pair_sum(uint32_t taddr, float (&v)[64]) {
  uint32_t h[32], l[32];
  tmem_ld32_nowait(taddr + J0, h);
  tmem_ld32_nowait(taddr + 64 + J0, l);
  tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < 32; ++j) v[J0 + j] = __uint_as_float(h[j]) + __uint_as_float(l[j]);
}

// ------------------------------------------------------------------ kernel
template <int D>
__global__ void __launch_bounds__(kAttThreads, 1)
    attention_tc_kernel(const __grid_constant__ AttMaps maps, const __grid_constant__ AttArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float *m_ref = reinterpret_cast<float *>(sm + kOffRed);  // per query: reference max (log2 units)
  float *alpha = m_ref + 64, *l_fin = alpha + 64;          // rescale factors, row sums
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
  uint64_t *full = bars, *empty = bars + 2, *sfull = bars + 4, *sfree = bars + 6;
  uint64_t *pfull = bars + 8, *pvdone = bars + 9, *qready = bars + 10;
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
  const int nt = n_ctx + (do_block ? 1 : 0);

  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(&empty[0], 1);
    mbar_init(&empty[1], 1);
    mbar_init(&sfull[0], 1);
    mbar_init(&sfull[1], 1);
    mbar_init(&sfree[0], kSoftThreads);
    mbar_init(&sfree[1], kSoftThreads);
    mbar_init(pfull, kSoftThreads);
    mbar_init(pvdone, 1);
    mbar_init(qready, kSoftThreads);
    *sabort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.ring_k);
    tma_prefetch_desc(&maps.ring_v);
    tma_prefetch_desc(&maps.blk_k);
    tma_prefetch_desc(&maps.blk_v);
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

  int issued = 0;
  if (warp == 0) {
    if (lane == 0) att_producer<D>(maps, a, sm, full, empty, b, g, F, t_begin, n_ctx, nt, sabort, issued);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) att_mma<D>(sm, full, empty, sfull, sfree, pfull, pvdone, qready, tmem, n_ctx, nt, sabort);
    __syncwarp();
  } else {
    const int qd = warp & 3;           // TMEM lane quarter of this warp
    const int kr = qd * 32 + lane;     // S^T lane = key row of a tile; O^T lane = output dim
    const int st_id = tid - 64;        // 0..127 among the softmax threads
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    pdl_wait();
    // Query tile: row n = plane*64 + r, r = head_in_group * W + i, plane 0 = hi, 1 = lo
    {
      const int n = st_id, plane = n >> 6, r = n & 63;
      const bool ok = r < R;
      const int hh = ok ? r / W : 0, i = ok ? r % W : 0;
      const uint4 *src = reinterpret_cast<const uint4 *>(
          static_cast<const __nv_bfloat16 *>(a.q) + (plane ? a.q_lo : 0) +
          (static_cast<size_t>(b) * W + i) * a.n_q_heads * D + static_cast<size_t>(g * G + hh) * D);
      uint4 v[D / 8];
#pragma unroll
      for (int ch = 0; ch < D / 8; ++ch) v[ch] = ok ? __ldg(src + ch) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int ch = 0; ch < D / 8; ++ch)
        *reinterpret_cast<uint4 *>(sm + kOffQ + (ch >> 3) * kAtom + n * 128 +
                                   (((ch & 7) ^ (n & 7)) << 4)) = v[ch];
    }
    if (st_id < 64) m_ref[st_id] = -INFINITY;
    fence_proxy_async_shared();
    mbar_arrive(qready);
    named_bar(kBarSoft, kSoftThreads);

    const float sl2 = 1.4426950408889634f * rsqrtf(static_cast<float>(D));  // log2(e)/sqrt(D)
    float lsum[64];
#pragma unroll
    for (int q = 0; q < 64; ++q) lsum[q] = 0.f;
    bool abort = false;
    for (int t = 0; t < nt && !abort; ++t) {
      const int sb = t & 1;
      bool ok = !*sabort && mbar_wait(&sfull[sb], (t >> 1) & 1);
      if (named_bar_or(kBarVote, kSoftThreads, !ok)) {
        abort = true;
        break;
      }
      tc_fence_after();
      float s[64];
      tmem_pair_sum<0>(tmem + lane_off + sb * 128, s);
      tmem_pair_sum<32>(tmem + lane_off + sb * 128, s);
      tc_fence_before();
      mbar_arrive(&sfree[sb]);  // the S buffer may take the tile after next
      const bool blk = t >= n_ctx;
      if (blk && qd == 0) {  // add the lo key rows (lanes 16..31) to their hi rows
#pragma unroll
        for (int q = 0; q < 64; ++q) s[q] += __shfl_down_sync(0xffffffffu, s[q], 16);
      }
      // visibility: context key at position p is seen by rows i <= i_max; block key kr by
      // rows i with the block rule
      int i_max = -1;
      if (!blk) {
        const int slot = (t_begin + t) * kTileKeys + kr;
        if (slot < n_slots) {
          const long long p = slot_position(F, cap, slot);
          if (a.window > 0) {
            const long long m = p - (F - a.window + 1);
            i_max = m < 0 ? -1 : (m > W ? W : static_cast<int>(m));
          } else {
            i_max = W;
          }
        }
      }
      bool need = false;
      {
        int i = 0;
#pragma unroll
        for (int q = 0; q < 64; ++q) {
          bool vis;
          if (!blk)
            vis = q < R && i <= i_max;
          else
            vis = q < R && kr < W && qd == 0 && (!a.causal || kr <= i) &&
                  (a.window <= 0 || abs(kr - i) < a.window);
          const float x = vis ? s[q] * sl2 : -INFINITY;
          s[q] = x;
          need |= x > m_ref[q] + 8.f;
          i = (i + 1 == W) ? 0 : i + 1;
        }
      }
      need = named_bar_or(kBarVote, kSoftThreads, need);
      // the previous tile's P.V has finished: the probability tile is free, O^T is stable
      ok = t == 0 || mbar_wait(pvdone, (t - 1) & 1);
      if (named_bar_or(kBarVote, kSoftThreads, !ok)) {
        abort = true;
        break;
      }
      if (need) {  // new reference maxima (exact over this tile), rescale l and O^T
        float *scr = reinterpret_cast<float *>(sm + kOffP);  // free: the last P.V is done
        table_store(scr, kr, s);
        named_bar(kBarSoft, kSoftThreads);
        if (st_id < 64) {
          const float tm = table_column<true>(scr, st_id);
          const float m_old = m_ref[st_id], m_new = fmaxf(m_old, tm);
          alpha[st_id] = m_new == -INFINITY ? 1.f : exp2f(m_old - m_new);
          m_ref[st_id] = m_new;
        }
        named_bar(kBarSoft, kSoftThreads);
#pragma unroll
        for (int q = 0; q < 64; ++q) lsum[q] *= alpha[q];
        if (t > 0) {  // O^T row kr: columns c and c + 64 belong to query c
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < 128; c0 += 32) {
            uint32_t o[32];
            tmem_ld32_nowait(tmem + lane_off + kTmemO + c0, o);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j)
              o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha[(c0 + j) & 63]);
            tmem_st32(tmem + lane_off + kTmemO + c0, o);
          }
          tmem_st_wait();
        }
      }
      // probabilities: bf16 hi and lo halves, key row kr of the P^T tile
      const bool dup = blk && qd == 0 && kr >= 16;  // block lo-key rows repeat rows 0..15
      if (!dup) {
        uint8_t *rowp = sm + kOffP + kr * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int q0 = c * 8 + 2 * e;
            const float p0 = s[q0] == -INFINITY ? 0.f : exp2f(s[q0] - m_ref[q0]);
            const float p1 = s[q0 + 1] == -INFINITY ? 0.f : exp2f(s[q0 + 1] - m_ref[q0 + 1]);
            lsum[q0] += p0;
            lsum[q0 + 1] += p1;
            const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
            const float2 hf = __bfloat1622float2(h);
            hw[e] = *reinterpret_cast<const uint32_t *>(&h);
            lw[e] = pack_bf16(p0 - hf.x, p1 - hf.y);
          }
          const uint32_t sw = static_cast<uint32_t>((c ^ (kr & 7)) << 4);
          *reinterpret_cast<uint4 *>(rowp + sw) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4 *>(rowp + kAtom + sw) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
      if (blk && qd == 0) {
        __syncwarp();
        if (dup) {  // same swizzle phase: kr & 7 == (kr - 16) & 7
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t o = static_cast<uint32_t>(c << 4);
            *reinterpret_cast<uint4 *>(sm + kOffP + kr * 128 + o) =
                *reinterpret_cast<const uint4 *>(sm + kOffP + (kr - 16) * 128 + o);
            *reinterpret_cast<uint4 *>(sm + kOffP + kAtom + kr * 128 + o) =
                *reinterpret_cast<const uint4 *>(sm + kOffP + kAtom + (kr - 16) * 128 + o);
          }
        }
      }
      fence_proxy_async_shared();
      tc_fence_before();
      mbar_arrive(pfull);
    }
    if (!abort && nt > 0) {
      const bool ok = mbar_wait(pvdone, (nt - 1) & 1);
      abort = named_bar_or(kBarVote, kSoftThreads, !ok);
    }
    if (!abort) {
      // row sums of the 128 threads' partial sums
      float *scr = reinterpret_cast<float *>(sm + kOffP);  // free: the last P.V is done
      table_store(scr, kr, lsum);
      named_bar(kBarSoft, kSoftThreads);
      if (st_id < 64) l_fin[st_id] = table_column<false>(scr, st_id);
      named_bar(kBarSoft, kSoftThreads);
      // O^T row kr (output dim d = kr): query q is columns q and q + 64
      float o[64];
      if (nt > 0) {
        tc_fence_after();
        tmem_pair_sum<0>(tmem + lane_off + kTmemO, o);
        tmem_pair_sum<32>(tmem + lane_off + kTmemO, o);
      } else {
#pragma unroll
        for (int q = 0; q < 64; ++q) o[q] = 0.f;
      }
      const size_t bh = static_cast<size_t>(b) * a.n_kv_heads + g;
      if (a.n_splits == 1) {
        if (kr < D) {
          __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out);
          int hh = 0, i = 0;
#pragma unroll
          for (int q = 0; q < 64; ++q) {
            if (q < R) {
              const float L = l_fin[q];
              const float y = L > 0.f ? o[q] / L : 0.f;
              const size_t idx = (static_cast<size_t>(b) * W + i) * a.n_q_heads * D +
                                 static_cast<size_t>(g * G + hh) * D + kr;
              const __nv_bfloat16 h = __float2bfloat16_rn(y);
              out[idx] = h;
              if (a.out_lo) out[a.out_lo + idx] = __float2bfloat16_rn(y - __bfloat162float(h));
            }
            if (++i == W) {
              i = 0;
              ++hh;
            }
          }
        }
      } else {
        float *po = a.part_o + (bh * a.n_splits + split) * kAttRows * D;
        if (kr < D) {
#pragma unroll
          for (int q = 0; q < 64; ++q) po[static_cast<size_t>(q) * D + kr] = o[q];
        }
        if (st_id < 64)
          a.part_ml[(bh * a.n_splits + split) * kAttRows + st_id] = make_float2(m_ref[st_id], l_fin[st_id]);
        // merge the splits in this launch: every split of (b, g) counts itself once its
        // partial is stored, waits (bounded) for the others, then merges its share of the
        // rows.  The launch has at most one CTA per SM, so all splits are resident together,
        // and each stores its partial before it waits.
        unsigned *arrived = a.counters + bh;
        unsigned *done = a.counters + static_cast<size_t>(a.B) * a.n_kv_heads + bh;
        __threadfence();
        named_bar(kBarSoft, kSoftThreads);
        bool wok = true;
        if (st_id == 0) {
          atomicAdd(arrived, 1u);
          wok = wait_count(arrived, static_cast<unsigned>(a.n_splits), kWaitLimitNs, 0);
        }
        if (!named_bar_or(kBarVote, kSoftThreads, !wok)) {
          const int rp = (R + a.n_splits - 1) / a.n_splits;
          const int r0 = min(R, split * rp), r1 = min(R, (split + 1) * rp);
          if (a.n_splits <= kFewSplits)
            combine_rows_few<__nv_bfloat16, D, kFewSplits, 2>(a, b, g, r0, r1, warp - 2, lane);
          else
            combine_rows<__nv_bfloat16, D>(a, b, g, r0, r1, warp - 2, lane,
                                           reinterpret_cast<float (*)[D + 4]>(sm + kOffP));
          named_bar(kBarSoft, kSoftThreads);
          if (st_id == 0 && atomicAdd(done, 1u) == static_cast<unsigned>(a.n_splits - 1)) {
            *arrived = 0u;  // every split is past its wait: ready for the next launch
            *done = 0u;
          }
        }
      }
    }
    if (abort) *sabort = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (*sabort && warp == 0 && lane == 0) {
    // a wait gave up: let the loads still in flight land before the CTA exits (bounded)
    for (int t = max(0, issued - 2); t < issued; ++t) mbar_wait(&full[t & 1], (t >> 1) & 1);
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

size_t attention_partial_floats(int B, int n_kv_heads, int n_splits, int head_dim) {
  return static_cast<size_t>(B) * n_kv_heads * n_splits * kAttRows * head_dim;
}
size_t attention_ml_count(int B, int n_kv_heads, int n_splits) {
  return static_cast<size_t>(B) * n_kv_heads * n_splits * kAttRows;
}
int attention_rows_max() { return kAttRows; }
int attention_tile_keys() { return kTileKeys; }

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
  return launch_pdl(attention_tc_kernel<D>, dim3(a.n_splits, a.n_kv_heads, a.B), dim3(kAttThreads),
                    kAttSmem, stream, m, a);
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
      !(err = make_tensor_map_2d(&m.blk_v, a.blk_v, GT_BF16, D, blk_rows, 64, 16, true)).empty())
    return err;
  e = D == 128 ? launch_tc<128>(m, a, stream) : launch_tc<64>(m, a, stream);
  if (e != cudaSuccess) return std::string("attention launch: ") + cudaGetErrorString(e);
  return {};
}

}  // namespace bd
