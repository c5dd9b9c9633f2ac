// Weight-streaming GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
//   D[tok, row] = sum_k X[tok, k] * W[row, k]
//
// Swap-AB: a 128-row weight tile is the MMA's A operand (M = 128), the token rows of the
// drafter block are the B operand (N = block_n <= 256, a multiple of 16).  Both operands
// are K-major tiles that TMA writes into shared memory with 128-byte swizzling; the fp32
// accumulator lives in tensor memory and is read back by four epilogue warps.
//
// Work split (stream-K): the (tile, k-block) units of all segments are cut into n_ctas
// contiguous ranges of equal length, so every SM streams the same number of weight bytes
// whatever the matrix shapes.  The CTAs that share a tile store fp32 partial tiles and,
// after their own mainloops, each sums a share of the tile over all partials in CTA
// order, so results do not depend on arrival order.  These are the only waits between
// CTAs; a launch never has more CTAs than SMs.
//
// Warp roles: warp 0 = TMA producer (one lane), warp 1 = TMEM owner and MMA issuer (one
// lane), warps 2-5 = epilogue (128 threads, one accumulator row each).
#include "bd_device.cuh"

#include <type_traits>
#include "bd_internal.h"

#include <cstdio>
#include <cstring>
#include <mutex>
#include <unordered_map>

namespace bd {

BD_DEFINE_ERROR_TAKER(take_error_word_gemm)

template <typename T> struct MmaTraits;
// kind: 0 = kind::f16 (fmt 0 fp16, 1 bf16), 1 = kind::tf32, 2 = kind::f8f6f4 (fmt 0 E4M3)
template <> struct MmaTraits<__nv_bfloat16> {
  static constexpr int BK = 64;   // k elements per 128-byte smem row
  static constexpr int UK = 16;   // k per tcgen05.mma
  static constexpr uint32_t fmt = 1;
  static constexpr int kind = 0;
};
template <> struct MmaTraits<__half> {
  static constexpr int BK = 64;
  static constexpr int UK = 16;
  static constexpr uint32_t fmt = 0;
  static constexpr int kind = 0;
};
template <> struct MmaTraits<float> {
  static constexpr int BK = 32;
  static constexpr int UK = 8;
  static constexpr uint32_t fmt = 2;
  static constexpr int kind = 1;
};
template <> struct MmaTraits<Fp8E4M3> {
  static constexpr int BK = 128;
  static constexpr int UK = 32;
  static constexpr uint32_t fmt = 0;
  static constexpr int kind = 2;
};

constexpr int kATileBytes = kBM * 128;  // 16 KB: 128 rows x 128 bytes
constexpr int kXStride = 17;            // epilogue exchange row stride (floats)
constexpr int kMaxStages = 12;
constexpr long long kMinUnits = 8;
constexpr double kWholeTileSlack = 1.15;
constexpr size_t kSmemLimit = 232448 - 1024;  // 227 KB opt-in per block, less static smem
// Products of up to 128 tokens whose weights are small (re-read from L2 at little cost) and
// fill at most half the SMs with 128-token tiles take tiles of kSmallBlockN tokens: twice the
// tiles, so more SMs share the weights and each tile's epilogue is half as long (the
// DSpine bridge's code read, gate maps and write at 128 tokens: 20 us less per 5-layer round).
constexpr int kSmallBlockN = 64;
constexpr long long kSmallWeightBytes = 12ll << 20;

// A pipeline stage holds kbox K-boxes of the weight tile (each 128 rows x 128 bytes, so
// every weight row is read in kbox*128-byte contiguous pieces) and the matching kbox
// boxes of the activation tile.
constexpr int kOutStage = 16 * kBM * 4;  // 8 KB: one 16-column chunk of fp32 results

// Stage area (the pipeline), then the epilogue's buffers: exchange, two output staging
// buffers, argmax scratch, INJECT row scales, barriers.
struct SmemLayout {
  size_t off_b, off_x, off_out, off_red, off_rs, off_bar, total;
};
__host__ __device__ inline SmemLayout smem_layout(int stages, int block_n, int kbox) {
  SmemLayout L;
  L.off_b = static_cast<size_t>(stages) * kbox * kATileBytes;
  L.off_x = L.off_b + static_cast<size_t>(stages) * kbox * block_n * 128;
  L.off_out = (L.off_x + kBM * kXStride * 4 + 1023) / 1024 * 1024;
  L.off_red = L.off_out + 2 * kOutStage;
  L.off_rs = L.off_red + 2 * (kEpiThreads / 2) * 4;  // maxima and indices, 16 per warp
  L.off_bar = L.off_rs + 256 * 4;
  L.total = L.off_bar + (2 * stages + 5) * 8 + 16 + 1024;  // + alignment slack
  return L;
}

// Walks the (tile, k-block range) segments of one CTA's stream-K unit range.
struct SegWalk {
  long long u, u1;
  int kb;
  __device__ bool next(int &tile, int &kb0, int &kb1) {
    if (u >= u1) return false;
    tile = static_cast<int>(u / kb);
    kb0 = static_cast<int>(u % kb);
    const long long rem = u1 - u;
    kb1 = static_cast<int>(rem < (kb - kb0) ? kb0 + rem : kb);
    u += kb1 - kb0;
    return true;
  }
};

// CTA c's units start at unit_begin(c): the U units are cut into grains of g units (1, or
// the k-blocks of a whole tile when every CTA takes whole tiles) dealt out evenly.
__device__ __forceinline__ long long unit_begin(long long U, int P, int c, int g) {
  return static_cast<long long>(c) * (U / g) / P * g;
}
// CTA whose unit range contains unit u.
__device__ __forceinline__ int cta_of_unit(long long U, int P, long long u, int g) {
  return static_cast<int>(((u / g + 1) * P - 1) / (U / g));
}

__device__ __forceinline__ int seg_of_tile(const GemmArgs &p, int m_tile) {
  int s = 0;
#pragma unroll 1
  for (int i = 1; i < p.n_segs; ++i)
    if (m_tile >= p.seg[i].tile_begin) s = i;
  return s;
}

// ------------------------------------------------------------------ producer
template <typename T>
__device__ void gemm_producer(const GemmMaps &maps, const GemmArgs &p, uint8_t *sA,
                              uint8_t *sB, uint64_t *full, uint64_t *empty, long long u0,
                              long long u1, volatile int *sabort) {
  constexpr int BK = MmaTraits<T>::BK;
  const uint64_t pol_w = policy_evict_first();
  const uint64_t pol_x = policy_evict_last();
  const int S = p.stages;
  const int KB = p.kbox;
  const uint32_t box_b = static_cast<uint32_t>(p.block_n) * 128u;
  const uint32_t a_bytes = static_cast<uint32_t>(KB) * kATileBytes;
  const uint32_t b_bytes = static_cast<uint32_t>(KB) * box_b;
  const int n_boxes = (p.K + BK - 1) / BK;  // boxes that hold any of the K columns
  // Boxes of unit kbi that start inside K; a box past the end is neither loaded nor used.
  auto boxes = [&](int kbi) { return min(KB, n_boxes - kbi * KB); };
  auto unit_bytes = [&](int kbi) {
    return static_cast<uint32_t>(boxes(kbi)) * (kATileBytes + box_b);
  };

  // s: the tile's weight segment (looked up once per tile)
  auto load_a = [&](int m_tile, int s, int kbi, uint8_t *dst, uint64_t *bar) {
    const int nb = boxes(kbi);
    if (p.packed) {  // the unit's boxes are one contiguous piece of the packed image
      const GemmSeg &sg = p.seg[s];
      const size_t box0 = static_cast<size_t>(m_tile - sg.tile_begin) * sg.n_kb_pack +
                          static_cast<size_t>(kbi) * KB;
      bulk_load(dst, sg.packed + box0 * kATileBytes, static_cast<uint32_t>(nb) * kATileBytes, bar,
                pol_w);
      return;
    }
    for (int j = 0; j < nb; ++j) {
      const int x = (kbi * KB + j) * BK;
      uint8_t *d = dst + static_cast<size_t>(j) * kATileBytes;
      if (p.pair_mode) {
        tma_load_2d(d, &maps.a[0], bar, x, m_tile * 64, pol_w);
        tma_load_2d(d + 64 * 128, &maps.a[1], bar, x, m_tile * 64, pol_w);
      } else {
        tma_load_2d(d, &maps.a[s], bar, x, (m_tile - p.seg[s].tile_begin) * kBM, pol_w);
      }
    }
  };
  auto load_b = [&](int n_tile, int kbi, uint8_t *dst, uint64_t *bar) {
    const int nb = boxes(kbi);
    for (int j = 0; j < nb; ++j) {
      uint8_t *d = dst + static_cast<size_t>(j) * box_b;
      const int x = (kbi * KB + j) * BK;
      if (p.split) {  // [hi rows of the tile; lo rows of the tile]
        tma_load_2d(d, &maps.b, bar, x, n_tile * p.ln, pol_x);
        tma_load_2d(d + static_cast<size_t>(p.ln) * 128, &maps.b, bar, x, p.lo_row + n_tile * p.ln,
                    pol_x);
      } else {
        tma_load_2d(d, &maps.b, bar, x, n_tile * p.block_n, pol_x);
      }
    }
  };

  // The weight tiles do not depend on the previous kernel: start streaming them before
  // waiting for it (programmatic dependent launch).
  const long long total = u1 - u0;
  const int pre = static_cast<int>(total < S ? total : S);
  {
    SegWalk w{u0, u1, p.kb};
    int tile, kb0, kb1, q = 0;
    while (q < pre && w.next(tile, kb0, kb1)) {
      const int m_tile = tile / p.n_tiles_n;
      const int sg = p.pair_mode ? 0 : seg_of_tile(p, m_tile);
      for (int kbi = kb0; kbi < kb1 && q < pre; ++kbi, ++q) {
        mbar_arrive_expect_tx(&full[q], unit_bytes(kbi));
        load_a(m_tile, sg, kbi, sA + static_cast<size_t>(q) * a_bytes, &full[q]);
      }
    }
  }
  pdl_wait();
  SegWalk w{u0, u1, p.kb};
  int tile, kb0, kb1;
  // stage s of pass `round` over the ring (counted incrementally: no division per stage)
  int q = 0, s = 0;
  uint32_t round = 0;
  while (w.next(tile, kb0, kb1)) {
    const int m_tile = tile / p.n_tiles_n, n_tile = tile % p.n_tiles_n;
    const int sg = p.pair_mode ? 0 : seg_of_tile(p, m_tile);
    for (int kbi = kb0; kbi < kb1; ++kbi) {
      if (q >= pre) {
        if (*sabort || !mbar_wait(&empty[s], (round & 1u) ^ 1u)) {
          *sabort = 1;
          return;
        }
        mbar_arrive_expect_tx(&full[s], unit_bytes(kbi));
        load_a(m_tile, sg, kbi, sA + static_cast<size_t>(s) * a_bytes, &full[s]);
      } else {
        ++q;
      }
      load_b(n_tile, kbi, sB + static_cast<size_t>(s) * b_bytes, &full[s]);
      if (++s == S) {
        s = 0;
        ++round;
      }
    }
  }
}

// ------------------------------------------------------------------ MMA issuer
template <typename T>
__device__ void gemm_mma(const GemmArgs &p, uint8_t *sA, uint8_t *sB, uint64_t *full,
                         uint64_t *empty, uint64_t *accf, uint64_t *acce, uint32_t tmem_base,
                         long long u0, long long u1, volatile int *sabort) {
  constexpr int BK = MmaTraits<T>::BK, UK = MmaTraits<T>::UK;
  const uint32_t idesc = umma_idesc(MmaTraits<T>::fmt, kBM, p.block_n);
  const int S = p.stages;
  const int KB = p.kbox;
  const uint32_t box_b = static_cast<uint32_t>(p.block_n) * 128u;
  const uint32_t a_bytes = static_cast<uint32_t>(KB) * kATileBytes;
  const uint32_t b_bytes = static_cast<uint32_t>(KB) * box_b;
  const int n_boxes = (p.K + BK - 1) / BK;
  SegWalk w{u0, u1, p.kb};
  int tile, kb0, kb1, e = 0;
  int s = 0;           // stage of the next unit
  uint32_t phase = 0;  // parity of its pass over the ring
  while (w.next(tile, kb0, kb1)) {
    const int a = e & 1;
    const uint32_t ra = static_cast<uint32_t>(e >> 1);
    if (*sabort || !mbar_wait(&acce[a], (ra & 1u) ^ 1u)) {
      *sabort = 1;
      return;
    }
    tc_fence_after();
    const uint32_t d = tmem_base + static_cast<uint32_t>(a * p.block_n);
    for (int kbi = kb0; kbi < kb1; ++kbi) {
      if (*sabort || !mbar_wait(&full[s], phase)) {
        *sabort = 1;
        return;
      }
      tc_fence_after();
      const uint32_t abase = smem_u32(sA + static_cast<size_t>(s) * a_bytes);
      const uint32_t bbase = smem_u32(sB + static_cast<size_t>(s) * b_bytes);
      const int nb = min(KB, n_boxes - kbi * KB);
      for (int j = 0; j < nb; ++j) {
#pragma unroll
        for (int k = 0; k < BK / UK; ++k) {
          const uint64_t ad = umma_desc_sw128(abase + j * kATileBytes + k * 32);
          const uint64_t bd = umma_desc_sw128(bbase + j * box_b + k * 32);
          const uint32_t acc = (kbi > kb0 || j > 0 || k > 0) ? 1u : 0u;
          if constexpr (MmaTraits<T>::kind == 0)
            umma_bf16(d, ad, bd, idesc, acc);  // kind::f16 (the idesc selects bf16 / fp16)
          else if constexpr (MmaTraits<T>::kind == 1)
            umma_tf32(d, ad, bd, idesc, acc);
          else
            umma_f8(d, ad, bd, idesc, acc);
        }
      }
      umma_commit(&empty[s]);  // the stage is free once these MMAs have read it
      if (++s == S) {
        s = 0;
        phase ^= 1u;
      }
    }
    umma_commit(&accf[a]);     // accumulator ready for the epilogue
    ++e;
  }
}

// ------------------------------------------------------------------ epilogue
// Each epilogue thread owns accumulator row r (its warp's TMEM lane quarter) and kCW of
// the 16 token columns of a chunk, starting at column c0 of the chunk.
constexpr int kCW = 16 / kEpiSlices;
struct EpiPos {
  int r;   // tile row 0..127
  int et;  // 0..kEpiThreads-1 among the epilogue threads
  int c0;  // first column of this thread's slice of a chunk
};

// Up to four 16-column chunks of the accumulator at once: the kCW columns col + 16 i ..
// + kCW - 1 (i < nc) of this thread's row go to v[kCW i ..], each the hi half plus, when the
// activation operand is split, the lo half that sits LW columns further.  One wait covers
// all the loads of a group of four.
__device__ __forceinline__ void tmem_ld_chunks(uint32_t tbase, int col, int LW, int split, int nc,
                                               float (&v)[4 * kCW]) {
  static_assert(kCW == 8, "tmem_ld_chunks loads 8 columns per chunk and thread");
  const uint32_t t = tbase + static_cast<uint32_t>(col);
  if (nc == 4) {
    tmem_ld8x4(t, t + 16, t + 32, t + 48, v);
    if (split) {
      float w[4 * kCW];
      tmem_ld8x4(t + LW, t + LW + 16, t + LW + 32, t + LW + 48, w);
#pragma unroll
      for (int i = 0; i < 4 * kCW; ++i) v[i] += w[i];
    }
    return;
  }
#pragma unroll
  for (int c = 0; c < 3; ++c) {
    if (c >= nc) break;
    float h[kCW];
    tmem_ld8(t + 16 * c, h);
    if (split) {
      float w[kCW];
      tmem_ld8(t + LW + 16 * c, w);
#pragma unroll
      for (int jj = 0; jj < kCW; ++jj) h[jj] += w[jj];
    }
#pragma unroll
    for (int jj = 0; jj < kCW; ++jj) v[c * kCW + jj] = h[jj];
  }
}

// Chunk c (0..3, at run time) of a group loaded by tmem_ld_chunks, without indexing the
// register array by a run-time value.
__device__ __forceinline__ void chunk_of(const float (&v4)[4 * kCW], int c, float (&v)[kCW]) {
#pragma unroll
  for (int jj = 0; jj < kCW; ++jj)
    v[jj] = c == 0 ? v4[jj] : c == 1 ? v4[kCW + jj] : c == 2 ? v4[2 * kCW + jj] : v4[3 * kCW + jj];
}

// Results leave the SM through shared memory: the epilogue threads write a chunk of 16
// token columns into one of two staging buffers and one thread hands it to TMA (a tiled
// store, an in-L2 reduce-add, or a contiguous bulk store), so no thread waits for write
// acknowledgements.
struct EpiSmem {
  uint8_t *out;    // [2][kOutStage] staging buffers
  int next;        // buffer the next chunk uses
  float *xbuf;     // [128][kXStride] exchange / transpose buffer
  float *red;      // [kEpiThreads / 32][16] per-warp column maxima
  int32_t *redi;   // [kEpiThreads / 32][16] their indices
  float *rs;       // [256] INJECT row scales of the current tile's tokens
};

// Claims the next staging buffer: the bulk group that last read it (two chunks ago) must
// have finished reading.  Ends with a barrier of the epilogue threads.
__device__ __forceinline__ uint8_t *stage_claim(EpiSmem &es, int et) {
  uint8_t *sb = es.out + es.next * kOutStage;
  es.next ^= 1;
  if (et == 0) bulk_wait_read<1>();
  named_bar(1, kEpiThreads);
  return sb;
}
// Publishes the staged chunk to the async proxy; thread et == 0 then issues the copy.
__device__ __forceinline__ void stage_publish() {
  fence_proxy_async_shared();
  named_bar(1, kEpiThreads);
}

// Per-(vocab tile, token) maximum and its lowest index: the chunk is transposed through
// shared memory so that each thread scans a group of rows of one column serially (rows
// in ascending order, so a strict comparison keeps the lowest index), then the row
// groups are merged within warps and across warps.
__device__ __forceinline__ void argmax_chunk(const GemmArgs &p, int m_tile, int tok0,
                                             const EpiPos &ps, const float (&v)[kCW],
                                             EpiSmem &es) {
  constexpr int kWarps = kEpiThreads / 32;
  constexpr int kRowsPerGroup = kBM * 16 / kEpiThreads;  // 8 rows per thread
  const int row_id = m_tile * kBM + ps.r;
  const float ws = p.wscale != nullptr && row_id < p.vocab ? p.wscale[row_id] : 1.f;
#pragma unroll
  for (int jj = 0; jj < kCW; ++jj)
    es.xbuf[ps.r * kXStride + ps.c0 + jj] = row_id < p.vocab ? v[jj] * ws : -INFINITY;
  named_bar(1, kEpiThreads);
  const int col = ps.et & 15, grp = ps.et >> 4;
  float best = -INFINITY;
  int bi = 0x7fffffff;
#pragma unroll
  for (int i = 0; i < kRowsPerGroup; ++i) {
    const int row = grp * kRowsPerGroup + i;
    const float x = es.xbuf[row * kXStride + col];
    if (x > best) {
      best = x;
      bi = m_tile * kBM + row;
    }
  }
  const float ob = __shfl_xor_sync(0xffffffffu, best, 16);
  const int oi = __shfl_xor_sync(0xffffffffu, bi, 16);
  if (ob > best || (ob == best && oi < bi)) {
    best = ob;
    bi = oi;
  }
  if ((ps.et & 31) < 16) {
    es.red[(ps.et >> 5) * 16 + col] = best;
    es.redi[(ps.et >> 5) * 16 + col] = bi;
  }
  named_bar(1, kEpiThreads);
  if (ps.et < 16) {
    float b = es.red[ps.et];
    int i = es.redi[ps.et];
    for (int w = 1; w < kWarps; ++w) {
      const float x = es.red[w * 16 + ps.et];
      const int xi = es.redi[w * 16 + ps.et];
      if (x > b || (x == b && xi < i)) {
        b = x;
        i = xi;
      }
    }
    const int tok = tok0 + ps.et;
    if (tok < p.n_tokens) {
      p.amax_val[static_cast<size_t>(m_tile) * p.n_tokens + tok] = b;
      p.amax_idx[static_cast<size_t>(m_tile) * p.n_tokens + tok] = i;
    }
  }
}

// (score, id) order of the candidate lists: higher score first, equal scores lower id first.

// Per-(vocab tile, token) 16 best rows, in candidate order.  The chunk is transposed
// through shared memory; the 16 threads of a half warp own one token column, 8 rows each,
// sorted locally; 16 rounds of a half-warp argmax over the list heads then give the
// column's candidates in order (the winning thread drops its head).  The lists are staged
// in shared memory and leave as two contiguous bulk stores per chunk.
__device__ __forceinline__ void topk_chunk(const GemmArgs &p, int m_tile, int tok0,
                                           const EpiPos &ps, const float (&v)[kCW],
                                           EpiSmem &es) {
  static_assert(kEpiThreads == 256, "16 token columns x 16 threads per column");
  const int row_id = m_tile * kBM + ps.r;
  const float ws = p.wscale != nullptr && row_id < p.vocab ? p.wscale[row_id] : 1.f;
#pragma unroll
  for (int jj = 0; jj < kCW; ++jj)
    es.xbuf[ps.r * kXStride + ps.c0 + jj] = row_id < p.vocab ? v[jj] * ws : -INFINITY;
  uint8_t *sb = stage_claim(es, ps.et);  // also orders the transpose writes before the reads
  float *sv = reinterpret_cast<float *>(sb);                 // [16 tokens][kTopK]
  int32_t *si = reinterpret_cast<int32_t *>(sb + 16 * kTopK * 4);
  const int col = ps.et >> 4, l16 = ps.et & 15;
  float lv[8];
  int li[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = l16 * 8 + i;
    lv[i] = es.xbuf[row * kXStride + col];
    li[i] = m_tile * kBM + row;
  }
#pragma unroll
  for (int i = 1; i < 8; ++i)
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
  for (int rnd = 0; rnd < kTopK; ++rnd) {
    float bv = lv[0];
    int bi = li[0];
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (cand_better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (li[0] == bi) {  // this thread's head was taken
#pragma unroll
      for (int i = 0; i < 7; ++i) {
        lv[i] = lv[i + 1];
        li[i] = li[i + 1];
      }
      lv[7] = -INFINITY;
      li[7] = 0x7fffffff;
    }
    if (l16 == 0) {
      sv[col * kTopK + rnd] = bv;
      si[col * kTopK + rnd] = bi;
    }
  }
  stage_publish();  // also frees the transpose buffer for the next chunk
  const int n_tok = min(16, p.n_tokens - tok0);
  if (ps.et == 0 && n_tok > 0) {
    const size_t o = (static_cast<size_t>(m_tile) * p.n_tokens + tok0) * kTopK;
    bulk_store(p.topk_val + o, sv, static_cast<uint32_t>(n_tok) * kTopK * 4);
    bulk_store(p.topk_idx + o, si, static_cast<uint32_t>(n_tok) * kTopK * 4);
    bulk_commit();
  }
}

// EPI_QKV, one 16-column chunk of a 128-row tile (one head of D = 128, two of D = 64).  The
// chunk is exchanged through shared memory; thread et then takes token column et / 16 and
// the eight rows (head dims) 8 (et % 16) .. + 7, so the D / 8 threads of a head are adjacent
// lanes of one half-warp: the head's sum of squares is a shuffle tree over them and the RoPE
// partner of dim d (d +- D/2) sits D / 16 lanes away.
__device__ __forceinline__ float qkv_gain(const QkvPost &h, const void *g, int d) {
  return h.out_f32 ? static_cast<const float *>(g)[d]
                   : __bfloat162float(static_cast<const __nv_bfloat16 *>(g)[d]);
}
__device__ __forceinline__ void qkv_chunk(const GemmArgs &p, int m_tile, int tok0,
                                          const EpiPos &ps, const float (&v)[kCW], EpiSmem &es) {
  const QkvPost &h = p.qkv;
#pragma unroll
  for (int jj = 0; jj < kCW; ++jj) es.xbuf[ps.r * kXStride + ps.c0 + jj] = v[jj];
  named_bar(1, kEpiThreads);
  const int c = ps.et >> 4, row0 = (ps.et & 15) * 8;
  float x[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) x[i] = es.xbuf[(row0 + i) * kXStride + c];
  named_bar(1, kEpiThreads);  // the exchange buffer is free for the next chunk
  const int s = seg_of_tile(p, m_tile);  // 0: queries, 1: keys, 2: values
  const int D = h.D, half = D / 2;
  const int head = (m_tile - p.seg[s].tile_begin) * (kBM / D) + row0 / D;
  const int d0 = row0 % D;
  const int tok = tok0 + c;
  const bool live = tok < p.n_tokens;
  if (s != 2) {  // every lane takes part in the shuffles, live or not
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) ss += x[i] * x[i];
    for (int o = 1; o < D / 8; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = rsqrtf(ss / static_cast<float>(D) + h.eps);
    const void *gn = s == 0 ? h.q_norm : h.k_norm;
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] *= inv * qkv_gain(h, gn, d0 + i);
    const float2 *cs = h.rope + static_cast<size_t>(live ? tok : 0) * half;
    float pv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) pv[i] = __shfl_xor_sync(0xffffffffu, x[i], D / 16);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int d = d0 + i;
      const float2 cr = cs[d % half];
      x[i] = d < half ? x[i] * cr.x - pv[i] * cr.y : x[i] * cr.x + pv[i] * cr.y;
    }
  }
  // a padding head of a partial last tile (D = 64 with an odd head count) is not stored
  if (!live || head >= (s == 0 ? h.n_q_heads : h.n_kv_heads)) return;
  size_t o, lo;
  void *dst;
  if (tok < h.T) {  // block row b * W + i
    if (s == 0) {
      o = static_cast<size_t>(tok) * h.n_q_heads * D + static_cast<size_t>(head) * D;
      dst = h.q;
      lo = h.q_lo;
      if (h.q_scale != 0.f)
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] *= h.q_scale;
    } else {
      const int b = tok / h.W, i = tok % h.W;
      o = ((static_cast<size_t>(b) * h.n_kv_heads + head) * h.W + i) * D;
      dst = s == 1 ? h.kblk : h.vblk;
      lo = h.kv_lo;
    }
  } else {  // pending context row: its key and value to the ring, if its position is live
    if (s == 0) return;
    const int rr = tok - h.T;
    const int req = h.row_req[rr];
    const long long pos = h.row_pos[rr];
    if (req < 0 || req >= h.n_req || pos < 0) {
      atomicOr(&g_error_word, DEVERR_BAD_INDEX);
      return;
    }
    const long long F = h.frontier[req];
    if (h.min_back > 0 && (pos < F - h.min_back || pos >= F)) {
      atomicOr(&g_error_word, DEVERR_BAD_INDEX);
      return;
    }
    if (pos < F - h.cap || pos >= F) return;  // outside the final live window
    o = ((static_cast<size_t>(req) * h.n_kv_heads + head) * h.cap + pos % h.cap) * D;
    dst = s == 1 ? h.kring : h.vring;
    lo = 0;
  }
  o += d0;
  if (h.out_f32) {
    float4 *f = reinterpret_cast<float4 *>(static_cast<float *>(dst) + o);
    f[0] = make_float4(x[0], x[1], x[2], x[3]);
    f[1] = make_float4(x[4], x[5], x[6], x[7]);
  } else {
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 hv = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
      const float2 hf = __bfloat1622float2(hv);
      const __nv_bfloat162 lv = __floats2bfloat162_rn(x[2 * i] - hf.x, x[2 * i + 1] - hf.y);
      hw[i] = *reinterpret_cast<const uint32_t *>(&hv);
      lw[i] = *reinterpret_cast<const uint32_t *>(&lv);
    }
    __nv_bfloat16 *bd = static_cast<__nv_bfloat16 *>(dst) + o;
    *reinterpret_cast<uint4 *>(bd) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    if (lo) *reinterpret_cast<uint4 *>(bd + lo) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
}

// Writes the finished values v (tile row ps.r, token columns tok0+ps.c0 .. +kCW-1; j0 =
// tok0 minus the tile's first token) of m_tile to the epilogue's destination.
template <typename T, int EPI>
__device__ __forceinline__ void emit_rows(const GemmMaps &maps, const GemmArgs &p, int m_tile,
                                          int tok0, int j0, const EpiPos &ps,
                                          const float (&v)[kCW], EpiSmem &es);
template <typename T, int EPI>
__device__ __forceinline__ void emit_chunk(const GemmMaps &maps, const GemmArgs &p, int m_tile,
                                           int tok0, int j0, const EpiPos &ps,
                                           const float (&v)[kCW], EpiSmem &es) {
  if constexpr (EPI == EPI_ARGMAX) {
    argmax_chunk(p, m_tile, tok0, ps, v, es);
    return;
  } else if constexpr (EPI == EPI_QKV) {
    qkv_chunk(p, m_tile, tok0, ps, v, es);
    return;
  } else if constexpr (EPI == EPI_TOPK) {
    topk_chunk(p, m_tile, tok0, ps, v, es);
    return;
  } else {
    emit_rows<T, EPI>(maps, p, m_tile, tok0, j0, ps, v, es);
  }
}

// The epilogues that write rows of results (stores, residual and injection adds, SwiGLU).
template <typename T, int EPI>
__device__ __forceinline__ void emit_rows(const GemmMaps &maps, const GemmArgs &p, int m_tile,
                                          int tok0, int j0, const EpiPos &ps,
                                          const float (&v)[kCW], EpiSmem &es) {
  const int r = ps.r, c0 = ps.c0;
  if (EPI == EPI_SWIGLU) {  // the chunk goes through the exchange buffer (see below)
#pragma unroll
    for (int jj = 0; jj < kCW; ++jj) es.xbuf[r * kXStride + c0 + jj] = v[jj];
  }
  uint8_t *sb = stage_claim(es, ps.et);
  if constexpr (EPI == EPI_SWIGLU) {
    // rows 0..63: gate features f, rows 64..127: up features f (same f); thread et takes
    // feature et % 64 of tokens 4 (et / 64) .. + 3
    static_assert(kEpiThreads == 256, "64 features x 4 token groups");
    T *hi = reinterpret_cast<T *>(sb);
    T *lo = hi + 16 * 64;
    const int f = ps.et & 63, cb = (ps.et >> 6) * 4;
    bool bad = false;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int c = cb + k;
      const float g = es.xbuf[f * kXStride + c], u = es.xbuf[(64 + f) * kXStride + c];
      const float h = __fdividef(g, 1.0f + __expf(-g)) * u;  // SiLU(g) u (-> 0 as g -> -inf)
      if constexpr (std::is_same<T, __half>::value) bad |= f16_out_of_range(h);
      const T hv = from_f<T>(h);
      hi[c * 64 + f] = hv;
      if (p.act_lo) lo[c * 64 + f] = from_f<T>(h - to_f<T>(hv));
    }
    flag_f16_range(bad);
  } else {
    float *f = reinterpret_cast<float *>(sb);
#pragma unroll
    for (int jj = 0; jj < kCW; ++jj) {
      const int c = c0 + jj;
      float x = v[jj];
      // anchor rows receive no write: adding -0 leaves every value bit-identical
      if (EPI == EPI_INJECT) x = ((tok0 + c) % p.block_w == 0) ? -0.0f : es.rs[j0 + c] * x;
      f[c * kBM + r] = x;
    }
  }
  stage_publish();
  if (ps.et == 0) {
    if (EPI == EPI_STORE_F32) {
      const int s = seg_of_tile(p, m_tile);
      tma_store_2d(&maps.out[s], sb, (m_tile - p.seg[s].tile_begin) * kBM, tok0);
    } else if (EPI == EPI_RESID_F32 || EPI == EPI_INJECT) {
      tma_reduce_add_2d(&maps.out[0], sb, m_tile * kBM, tok0);
    } else if (EPI == EPI_SWIGLU) {
      if (p.act_lo)
        tma_store_3d(&maps.out[0], sb, m_tile * 64, tok0, 0);
      else
        tma_store_2d(&maps.out[0], sb, m_tile * 64, tok0);
    }
    bulk_commit();
  }
}

// INJECT: row scales of the tile's tokens, read once per tile.  Safe to overwrite here:
// every thread has passed the barrier that ends the previous chunk's staging.
__device__ __forceinline__ void load_row_scales(const GemmArgs &p, int tile_tok0, int LW, int et,
                                                EpiSmem &es) {
  for (int t = et; t < LW; t += kEpiThreads) {
    const int tok = tile_tok0 + t;
    es.rs[t] = tok < p.n_tokens ? p.row_scale[tok] : 0.f;
  }
}

// Split tiles.  Every CTA that computed part of a tile stores its fp32 partial (layout
// [LW columns][128 rows], straight from registers: a warp writes 128 contiguous bytes per
// column) in its own slot (0 for the CTA's first tile, 1 for its last) and counts itself on
// the tile's counter.  After its mainloop each
// contributor waits until all n have arrived and then sums its share of the tile's
// 16-column chunks (chunk k belongs to the contributor k mod n) over all n partials, in CTA
// order, so results do not depend on which CTA got there first.  The partial values a
// thread adds (its row, its columns of the chunk) are loaded straight from L2, up to
// kFixLoads at a time before any of them is used.  Every contributor of a tile waits only
// for partials that the others write before their own waits, and all CTAs of a launch are
// resident at once (one per SM), so the waits end.
constexpr int kFixLoads = 32;

// The contributors of a split tile: CTAs c_first .. c_first + n - 1.  Each of them except
// c_first starts its unit range inside the tile, so the tile is its first (slot 0);
// c_first holds it in slot 1 when its range began in an earlier tile.  Worked out before
// the CTA's mainloop ends (the 64-bit divisions stay off the epilogue's critical path).
struct SplitInfo {
  int tile, c_first, n, slot0;
};
__device__ __forceinline__ SplitInfo split_info(const GemmArgs &p, int tile) {
  const long long U = p.units;
  const int P = p.n_ctas;
  const long long first_unit = static_cast<long long>(tile) * p.kb;
  SplitInfo si;
  si.tile = tile;
  si.c_first = cta_of_unit(U, P, first_unit, p.grain);
  si.n = cta_of_unit(U, P, first_unit + p.kb - 1, p.grain) - si.c_first + 1;
  si.slot0 = unit_begin(U, P, si.c_first, p.grain) < first_unit ? 1 : 0;
  return si;
}

template <typename T, int EPI>
__device__ bool fixup_tile(const GemmMaps &maps, const GemmArgs &p, const SplitInfo &si,
                           const EpiPos &ps, EpiSmem &es, volatile int *sabort) {
  const int tile = si.tile;
  const int LW = p.ln;
  const int m_tile = tile / p.n_tiles_n, n_tile = tile % p.n_tiles_n;
  const int c_first = si.c_first;
  const int n = si.n;
  const int me = static_cast<int>(blockIdx.x) - c_first;
  unsigned *arrived = p.counters + tile;
  unsigned *done = p.counters + p.n_counter_tiles + tile;
  const int n_chunks = LW / 16;
  const int my_chunks = me < n_chunks ? (n_chunks - me + n - 1) / n : 0;  // chunks me, me+n, ...
  const int et = ps.et;
  if (my_chunks > 0) {
    if (et == 0) {
      if (!wait_count(arrived, static_cast<unsigned>(n))) *sabort = 1;
    }
    named_bar(1, kEpiThreads);
    if (*sabort) return false;
    if (EPI == EPI_INJECT) load_row_scales(p, n_tile * LW, LW, et, es);
    // this thread's first value of chunk k in contributor i's partial
    auto src = [&](int i, int k) -> const float * {
      const int cslot = i == 0 ? si.slot0 : 0;
      return p.partials + (static_cast<size_t>(c_first + i) * 2 + cslot) * LW * kBM +
             static_cast<size_t>(k * 16 + ps.c0) * kBM + ps.r;
    };
    // one chunk at a time (one call site of the emit code: it is cold, once-per-tile code);
    // the contributors' values of a chunk are loaded G at a time before they are added
    constexpr int G = kFixLoads / kCW;
    for (int j = 0; j < my_chunks; ++j) {
      const int k = me + j * n;
      float acc[kCW];
#pragma unroll
      for (int jj = 0; jj < kCW; ++jj) acc[jj] = 0.f;
      for (int i0 = 0; i0 < n; i0 += G) {
        float v[G][kCW];
#pragma unroll
        for (int g = 0; g < G; ++g)
          if (i0 + g < n) {
            const float *sp = src(i0 + g, k);
#pragma unroll
            for (int jj = 0; jj < kCW; ++jj) v[g][jj] = __ldcg(sp + static_cast<size_t>(jj) * kBM);
          }
#pragma unroll
        for (int g = 0; g < G; ++g)
          if (i0 + g < n) {
#pragma unroll
            for (int jj = 0; jj < kCW; ++jj) acc[jj] += v[g][jj];
          }
      }
      emit_chunk<T, EPI>(maps, p, m_tile, n_tile * LW + k * 16, k * 16, ps, acc, es);
    }
  }
  if (et == 0) {
    if (atomicAdd(done, 1u) == static_cast<unsigned>(n - 1)) {  // every contributor is past its wait
      *arrived = 0u;
      *done = 0u;
    }
  }
  return true;
}

template <typename T, int EPI>
__device__ void gemm_epilogue(const GemmMaps &maps, const GemmArgs &p, uint64_t *accf,
                              uint64_t *acce, uint32_t tmem_base, long long u0, long long u1,
                              EpiSmem &es, volatile int *sabort) {
  const int warp = threadIdx.x >> 5;
  const int q = warp & 3;  // TMEM lane quarter this warp may access
  EpiPos ps;
  ps.r = q * 32 + (threadIdx.x & 31);
  ps.et = threadIdx.x - 64;
  ps.c0 = ((warp - 2) >> 2) * kCW;  // warps 2-5 take the first columns, 6-9 the next
  const int r = ps.r, et = ps.et;
  const int cta = blockIdx.x;
  const int first_tile = static_cast<int>(u0 / p.kb);
  // Only the first and the last tile of a CTA's unit range can be split.
  SplitInfo sp0{-1, 0, 0, 0}, sp1{-1, 0, 0, 0};
  {
    SegWalk sw{u0, u1, p.kb};
    int t, a0, a1;
    while (sw.next(t, a0, a1))
      if (a0 != 0 || a1 != p.kb) {
        if (sp0.tile < 0)
          sp0 = split_info(p, t);
        else
          sp1 = split_info(p, t);
      }
  }
  pdl_wait();
  SegWalk w{u0, u1, p.kb};
  int tile, kb0, kb1, e = 0;
  while (w.next(tile, kb0, kb1)) {
    const int a = e & 1;
    const uint32_t ra = static_cast<uint32_t>(e >> 1);
    ++e;
    const int m_tile = tile / p.n_tiles_n, n_tile = tile % p.n_tiles_n;
    const int LW = p.ln;  // logical token columns of the tile
    const bool whole = (kb0 == 0 && kb1 == p.kb);
    if (EPI == EPI_INJECT && whole) load_row_scales(p, n_tile * LW, LW, et, es);
    if (*sabort || !mbar_wait(&accf[a], ra & 1u)) {
      *sabort = 1;
      return;
    }
    tc_fence_after();
    const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                           static_cast<uint32_t>(a * p.block_n);
    if (!whole) {
      const int slot = (tile == first_tile) ? 0 : 1;
      float *mine = p.partials + (static_cast<size_t>(cta) * 2 + slot) * LW * kBM + r;
      for (int j0 = 0; j0 < LW; j0 += 64) {
        const int nc = min(4, (LW - j0) >> 4);
        float v4[4 * kCW];
        tmem_ld_chunks(tbase, j0 + ps.c0, LW, p.split, nc, v4);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (c < nc)
#pragma unroll
            for (int jj = 0; jj < kCW; ++jj)
              mine[static_cast<size_t>(j0 + 16 * c + ps.c0 + jj) * kBM] = v4[c * kCW + jj];
      }
      tc_fence_before();
      mbar_arrive(&acce[a]);  // the accumulator is free for the MMA warp
      // The barrier orders every thread's partial stores before thread 0's fence, which
      // makes them visible at device scope before the count.
      named_bar(1, kEpiThreads);
      if (et == 0) {
        __threadfence();
        atomicAdd(&p.counters[tile], 1u);
      }
      continue;
    }
    for (int j0 = 0; j0 < LW; j0 += 64) {
      const int nc = min(4, (LW - j0) >> 4);
      float v4[4 * kCW];
      tmem_ld_chunks(tbase, j0 + ps.c0, LW, p.split, nc, v4);
      if (j0 + 64 >= LW) {  // every column of the tile is in registers
        tc_fence_before();
        mbar_arrive(&acce[a]);
      }
      for (int c = 0; c < nc; ++c) {
        float v[kCW];
        chunk_of(v4, c, v);
        emit_chunk<T, EPI>(maps, p, m_tile, n_tile * LW + j0 + 16 * c, j0 + 16 * c, ps, v, es);
      }
    }
  }
  // The split tiles this CTA contributed to, reduced after its own mainloop.
  for (int i = 0; i < 2; ++i) {
    const SplitInfo si = i == 0 ? sp0 : sp1;
    if (si.tile < 0) break;
    if (!fixup_tile<T, EPI>(maps, p, si, ps, es, sabort)) {
      *sabort = 1;
      break;
    }
  }
  if (et == 0) bulk_wait<0>();  // every store of this CTA is complete before it exits
}

// ------------------------------------------------------------------ kernel
// One instantiation per (element type, epilogue): each kernel carries only the code of
// its own epilogue, which keeps the once-per-tile epilogue path small in the instruction
// cache.
template <typename T, int EPI>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ GemmMaps maps, const __grid_constant__ GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const SmemLayout L = smem_layout(p.stages, p.block_n, p.kbox);
  uint8_t *sA = smem;
  uint8_t *sB = smem + L.off_b;
  EpiSmem es;
  es.out = smem + L.off_out;
  es.next = 0;
  es.xbuf = reinterpret_cast<float *>(smem + L.off_x);
  es.red = reinterpret_cast<float *>(smem + L.off_red);
  es.redi = reinterpret_cast<int32_t *>(es.red + kEpiThreads / 2);
  es.rs = reinterpret_cast<float *>(smem + L.off_rs);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.off_bar);
  uint64_t *empty = full + p.stages;
  uint64_t *accf = empty + p.stages;
  uint64_t *acce = accf + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acce + 2);
  volatile int *sabort = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long u0 = unit_begin(p.units, p.n_ctas, blockIdx.x, p.grain);
  const long long u1 = unit_begin(p.units, p.n_ctas, blockIdx.x + 1, p.grain);
  uint32_t ncols = 32;
  while (ncols < static_cast<uint32_t>(2 * p.block_n)) ncols <<= 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&accf[0], 1);
    mbar_init(&accf[1], 1);
    mbar_init(&acce[0], kEpiThreads);
    mbar_init(&acce[1], kEpiThreads);
    *sabort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.b);
    if (!p.packed)
      for (int s = 0; s < (p.pair_mode ? 2 : p.n_segs); ++s) tma_prefetch_desc(&maps.a[s]);
  }
  if (threadIdx.x == 64) {  // result maps, used by the epilogue's stores
    const int n_out = EPI == EPI_STORE_F32 ? p.n_segs
                      : (EPI == EPI_ARGMAX || EPI == EPI_TOPK || EPI == EPI_QKV ? 0 : 1);
    for (int s = 0; s < n_out; ++s) tma_prefetch_desc(&maps.out[s]);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) gemm_producer<T>(maps, p, sA, sB, full, empty, u0, u1, sabort);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) gemm_mma<T>(p, sA, sB, full, empty, accf, acce, tmem_base, u0, u1, sabort);
    __syncwarp();
  } else {
    gemm_epilogue<T, EPI>(maps, p, accf, acce, tmem_base, u0, u1, es, sabort);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, ncols);
  }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

struct MapKey {
  const void *ptr;
  int dtype, inner, outer, box_inner, box_outer, swizzle, planes;
  long long stride, plane_stride;
  bool operator==(const MapKey &o) const {
    return ptr == o.ptr && dtype == o.dtype && inner == o.inner && outer == o.outer &&
           box_inner == o.box_inner && box_outer == o.box_outer && swizzle == o.swizzle &&
           stride == o.stride && planes == o.planes && plane_stride == o.plane_stride;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey &k) const {
    size_t h = std::hash<const void *>()(k.ptr);
    h ^= (static_cast<size_t>(k.inner) * 0x9E3779B97F4A7C15ull) + (h << 6) + (h >> 2);
    h ^= (static_cast<size_t>(k.outer) * 0xC2B2AE3D27D4EB4Full) + (h << 6) + (h >> 2);
    h ^= static_cast<size_t>(k.box_outer * 131 + k.box_inner * 7 + k.dtype * 3 + k.swizzle);
    h ^= (static_cast<size_t>(k.stride) * 0x165667B19E3779F9ull) + (h << 6) + (h >> 2);
    h ^= (static_cast<size_t>(k.plane_stride * 8 + k.planes) * 0x27D4EB2F165667C5ull) + (h << 6) +
         (h >> 2);
    return h;
  }
};

// Row-major [outer, inner] matrix (rows `stride` elements apart) -> 2-D tiled map with
// zero fill out of bounds; 128-byte swizzle for MMA operands, none for result tiles.
// planes > 1 adds a third dimension: `planes` such matrices plane_stride elements apart,
// all of them in every box.
static std::string make_map(CUtensorMap *out, const void *ptr, int dtype, int inner, int outer,
                            int box_inner, int box_outer, bool swizzle = true,
                            long long stride = 0, int planes = 1, long long plane_stride = 0) {
  static std::mutex mu;
  static std::unordered_map<MapKey, CUtensorMap, MapKeyHash> cache;
  if (stride == 0) stride = inner;
  const MapKey key{ptr,   dtype,          inner,  outer, box_inner, box_outer, swizzle ? 1 : 0,
                   planes, stride, plane_stride};
  {
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *out = it->second;
      return {};
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return "cuTensorMapEncodeTiled is unavailable";
  const int elem = (dtype == GT_BF16 || dtype == GT_F16) ? 2 : (dtype == GT_E4M3 ? 1 : 4);
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer),
                        static_cast<cuuint64_t>(planes)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(stride) * elem,
                           static_cast<cuuint64_t>(plane_stride) * elem};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer),
                       static_cast<cuuint32_t>(planes)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUtensorMap m;
  const CUtensorMapDataType ty = dtype == GT_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                 : dtype == GT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                 : dtype == GT_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  CUresult r = fn(&m, ty,
                  planes > 1 ? 3 : 2, const_cast<void *>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[160];
    snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d) for [%d x %d] box [%d x %d]",
             static_cast<int>(r), outer, inner, box_outer, box_inner);
    return buf;
  }
  {
    std::lock_guard<std::mutex> g(mu);
    cache[key] = m;
  }
  *out = m;
  return {};
}

std::string make_tensor_map_2d(CUtensorMap *out, const void *ptr, int dtype, int inner, int outer,
                               int box_inner, int box_outer, bool swizzle, long long stride) {
  return make_map(out, ptr, dtype, inner, outer, box_inner, box_outer, swizzle, stride);
}

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
  }
  return n;
}

int gemm_block_n(int n_tokens) {
  if (n_tokens <= 128) return ((n_tokens + 15) / 16) * 16;
  return 256;
}
int gemm_max_n_tiles(int n_tokens) { return (n_tokens + 15) / 16 * 16 / kSmallBlockN + 1; }

size_t gemm_partial_floats(int n_ctas, int block_n) {
  return static_cast<size_t>(n_ctas) * 2 * block_n * kBM;
}

// Deepest pipeline that fits in shared memory (0 if not even two stages fit).
static int pick_stages(int block_n, int kbox) {
  for (int s = kMaxStages; s >= 2; --s)
    if (smem_layout(s, block_n, kbox).total <= kSmemLimit) return s;
  return 0;
}

// K boxes per stage: as many as still leave a double-buffered pipeline (measured: two
// stages of 4 boxes, i.e. 512-byte row pieces, stream faster than deeper pipelines of
// narrower stages), and no more than half of K.
static int pick_kbox(int block_n, int K, int BK) {
  int kb = 4;
  while (kb > 1 && (pick_stages(block_n, kb) < 2 || K < kb * BK * 2)) kb >>= 1;
  return kb;
}

template <typename T, int EPI>
static cudaError_t launch_epi(const GemmMaps &maps, const GemmArgs &a, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<T, EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemLimit));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const size_t smem = smem_layout(a.stages, a.block_n, a.kbox).total;
  return launch_pdl(gemm_kernel<T, EPI>, dim3(a.n_ctas), dim3(kGemmThreads), smem, stream, maps,
                    a);
}

template <typename T>
static cudaError_t launch_typed(const GemmMaps &maps, const GemmArgs &a, cudaStream_t stream) {
  switch (a.epi) {
    case EPI_STORE_F32: return launch_epi<T, EPI_STORE_F32>(maps, a, stream);
    case EPI_RESID_F32: return launch_epi<T, EPI_RESID_F32>(maps, a, stream);
    case EPI_INJECT: return launch_epi<T, EPI_INJECT>(maps, a, stream);
    case EPI_SWIGLU: return launch_epi<T, EPI_SWIGLU>(maps, a, stream);
    case EPI_ARGMAX: return launch_epi<T, EPI_ARGMAX>(maps, a, stream);
    case EPI_TOPK: return launch_epi<T, EPI_TOPK>(maps, a, stream);
    case EPI_QKV: return launch_epi<T, EPI_QKV>(maps, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

std::string launch_gemm(GemmPlan &plan, const GemmScratch &sc, cudaStream_t stream) {
  GemmArgs &a = plan.args;
  const int BK = (plan.dtype == GT_BF16 || plan.dtype == GT_F16) ? 64
                 : (plan.dtype == GT_E4M3 ? 128 : 32);  // 128 bytes
  if (plan.n_tokens <= 0 || plan.K <= 0 || plan.n_w <= 0) return "empty GEMM";
  if (plan.n_w > kMaxSegs) return "too many GEMM segments";
  a.K = plan.K;
  a.n_tokens = plan.n_tokens;
  const int n_pad = (plan.n_tokens + 15) / 16 * 16;
  if (plan.split) {  // n-tiles of up to 128 tokens, each with its hi and lo rows
    if (plan.dtype != 0) return "split activations need bf16";
    a.split = 1;
    a.ln = n_pad <= 128 ? n_pad : 128;
    a.lo_row = n_pad;
    a.block_n = 2 * a.ln;
    a.n_tiles_n = (n_pad + a.ln - 1) / a.ln;
  } else {
    a.split = 0;
    a.block_n = gemm_block_n(plan.n_tokens);
    if (!plan.pair_mode && a.block_n > kSmallBlockN && a.block_n <= 128 && a.epi != EPI_ARGMAX &&
        a.epi != EPI_TOPK) {
      const int elem = (plan.dtype == GT_BF16 || plan.dtype == GT_F16) ? 2 : (plan.dtype == GT_E4M3 ? 1 : 4);
      long long mt = 0, wbytes = 0;
      for (int s = 0; s < plan.n_w; ++s) {
        mt += (plan.w[s].rows + kBM - 1) / kBM;
        wbytes += static_cast<long long>(plan.w[s].rows) * plan.K * elem;
      }
      if (2 * mt <= num_sms() && wbytes <= kSmallWeightBytes) a.block_n = kSmallBlockN;
    }
    a.ln = a.block_n;
    a.lo_row = 0;
    a.n_tiles_n = (plan.n_tokens + a.block_n - 1) / a.block_n;
  }
  a.pair_mode = plan.pair_mode ? 1 : 0;
  a.kbox = pick_kbox(a.block_n, plan.K, BK);
  a.kb = (plan.K + BK * a.kbox - 1) / (BK * a.kbox);
  int m_tiles = 0;
  if (plan.pair_mode) {
    if (plan.n_w != 2 || plan.w[0].rows != plan.w[1].rows) return "pair GEMM needs two equal matrices";
    a.n_segs = 1;
    a.seg[0].rows = plan.w[0].rows;
    a.seg[0].tile_begin = 0;
    m_tiles = (plan.w[0].rows + 63) / 64;
  } else {
    a.n_segs = plan.n_w;
    for (int s = 0; s < plan.n_w; ++s) {
      a.seg[s].rows = plan.w[s].rows;
      a.seg[s].tile_begin = m_tiles;
      m_tiles += (plan.w[s].rows + kBM - 1) / kBM;
    }
  }
  a.m_tiles = m_tiles;
  const long long tiles = static_cast<long long>(m_tiles) * a.n_tiles_n;
  a.units = tiles * a.kb;
  // Every CTA streams at least kMinUnits k-blocks (128 KB of weights): small matrices
  // use fewer CTAs instead of many tiny partial tiles.
  const long long min_units = (kMinUnits + a.kbox - 1) / a.kbox;
  const long long by_units = (a.units + min_units - 1) / min_units;
  a.n_ctas = static_cast<int>(by_units < num_sms() ? by_units : num_sms());
  // Whole tiles per CTA when there are at least as many tiles as CTAs and the busiest CTA
  // gets at most kWholeTileSlack times the average: no split tile, so no partial-tile
  // stores, waits or reductions (which cost more than that imbalance).
  a.grain = 1;
  if (tiles >= a.n_ctas) {
    const long long most = (tiles + a.n_ctas - 1) / a.n_ctas;
    if (static_cast<double>(most) * a.n_ctas <= kWholeTileSlack * static_cast<double>(tiles))
      a.grain = a.kb;
  }
  a.stages = pick_stages(a.block_n, a.kbox);
  if (a.stages < 2) return "GEMM tile does not fit in shared memory";
  a.partials = sc.partials;
  a.counters = sc.counters;
  a.n_counter_tiles = static_cast<int>(sc.n_counters);
  if (gemm_partial_floats(a.n_ctas, a.block_n) > sc.partial_floats) return "GEMM partial scratch too small";
  if (static_cast<size_t>(tiles) > sc.n_counters) return "GEMM counter scratch too small";

  GemmMaps maps;
  memset(&maps, 0, sizeof maps);
  a.packed = plan.w[0].packed != nullptr ? 1 : 0;
  if (a.packed) {
    const int elem = (plan.dtype == GT_BF16 || plan.dtype == GT_F16) ? 2 : (plan.dtype == GT_E4M3 ? 1 : 4);
    for (int s = 0; s < a.n_segs; ++s) {
      if (!plan.w[s].packed) return "packed GEMM with an unpacked segment";
      a.seg[s].packed = static_cast<const uint8_t *>(plan.w[s].packed);
      a.seg[s].n_kb_pack = static_cast<int>(packed_kb(plan.K, elem));
    }
  } else {
    if (plan.dtype == GT_E4M3 || plan.dtype == GT_F16) return "FP8 / fp16 GEMMs need packed weights";
    for (int s = 0; s < plan.n_w; ++s) {
      std::string err = make_map(&maps.a[s], plan.w[s].ptr, plan.dtype, plan.K, plan.w[s].rows, BK,
                                 plan.pair_mode ? 64 : kBM);
      if (!err.empty()) return err;
    }
  }
  std::string err = plan.split
      ? make_map(&maps.b, plan.x, plan.dtype, plan.K, 2 * a.lo_row, BK, a.ln)
      : make_map(&maps.b, plan.x, plan.dtype, plan.K, plan.n_tokens, BK, a.block_n);
  if (!err.empty()) return err;
  // Result maps: [n_tokens rows, output columns], boxes of 16 tokens.
  switch (a.epi) {
    case EPI_STORE_F32:
      for (int s = 0; s < a.n_segs && err.empty(); ++s)
        err = make_map(&maps.out[s], a.out_f32 + a.seg[s].out_col, 1, a.seg[s].rows, plan.n_tokens,
                       kBM, 16, false, a.ld_out);
      break;
    case EPI_RESID_F32:
    case EPI_INJECT:
      err = make_map(&maps.out[0], a.out_f32, 1, plan.w[0].rows, plan.n_tokens, kBM, 16, false,
                     a.ld_out);
      break;
    case EPI_SWIGLU:  // hi and lo planes (act_lo elements apart) in one box
      err = make_map(&maps.out[0], a.out_act, plan.dtype, plan.w[0].rows, plan.n_tokens, 64, 16,
                     false, a.ld_act, a.act_lo ? 2 : 1, a.act_lo);
      break;
    default:
      break;
  }
  if (!err.empty()) return err;
  cudaError_t e;
  if (plan.dtype == GT_E4M3) {
    if (a.epi != EPI_TOPK || plan.split || plan.pair_mode) return "FP8 GEMMs support the top-k epilogue only";
    e = launch_epi<Fp8E4M3, EPI_TOPK>(maps, a, stream);
  } else if (plan.dtype == GT_F16) {
    e = launch_typed<__half>(maps, a, stream);
  } else {
    e = plan.dtype == GT_BF16 ? launch_typed<__nv_bfloat16>(maps, a, stream)
                              : launch_typed<float>(maps, a, stream);
  }
  if (e != cudaSuccess) return std::string("GEMM launch: ") + cudaGetErrorString(e);
  return {};
}

}  // namespace bd
