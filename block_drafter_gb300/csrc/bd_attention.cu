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
  int p_lo, n_ctx, n_keys, k_begin, k_end;
};

__device__ __forceinline__ AttGeom att_geom(const AttArgs &a, int b, int split) {
  AttGeom g;
  g.F = a.frontier[b];
  long long lo = a.window > 0 ? g.F - a.window + 1 : 0;
  if (g.F - a.cap > lo) lo = g.F - a.cap;  // the ring holds [F - cap, F)
  if (lo < 0) lo = 0;
  g.p_lo = static_cast<int>(lo);
  g.n_ctx = static_cast<int>(g.F - lo);
  g.n_keys = g.n_ctx + a.W;
  int chunk = (g.n_keys + a.n_splits - 1) / a.n_splits;
  chunk = (chunk + kAttKeys - 1) / kAttKeys * kAttKeys;
  g.k_begin = split * chunk;
  g.k_end = min(g.n_keys, g.k_begin + chunk);
  return g;
}

// Is key k (0-based over [context; block]) visible from block row i?
__device__ __forceinline__ bool att_visible(const AttArgs &a, const AttGeom &g, int i, int k) {
  if (k >= g.k_end) return false;
  if (k < g.n_ctx) {
    const long long p = g.p_lo + k;
    return a.window <= 0 || (g.F + i) - p < a.window;
  }
  const int j = k - g.n_ctx;
  if (a.window > 0 && abs(j - i) >= a.window) return false;
  return !a.causal || j <= i;
}

template <int D>
__global__ void __launch_bounds__(128) attention_bf16_kernel(AttArgs a) {
  extern __shared__ uint8_t smem_raw[];
  constexpr int RS = D + kAttPad;  // smem row stride (elements)
  __nv_bfloat16 *sQ = reinterpret_cast<__nv_bfloat16 *>(smem_raw);
  __nv_bfloat16 *sK = sQ + kAttRows * RS;               // [2][kAttKeys][RS]
  __nv_bfloat16 *sV = sK + 2 * kAttKeys * RS;           // [2][kAttKeys][RS]

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.n_q_heads / a.n_kv_heads;
  const int R = G * a.W;
  pdl_wait();
  pdl_trigger();
  const AttGeom g = att_geom(a, b, split);

  const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q);
  const __nv_bfloat16 *ring_k = static_cast<const __nv_bfloat16 *>(a.ring_k);
  const __nv_bfloat16 *ring_v = static_cast<const __nv_bfloat16 *>(a.ring_v);
  const __nv_bfloat16 *blk_k = static_cast<const __nv_bfloat16 *>(a.blk_k);
  const __nv_bfloat16 *blk_v = static_cast<const __nv_bfloat16 *>(a.blk_v);

  // ---- Q tile: row rr = g_head * W + i  <-  q[(b*W + i), (h*G + g_head)*D + d]
  constexpr int CPR = D / 8;  // 16-byte chunks per row
  for (int c = tid; c < kAttRows * CPR; c += 128) {
    const int rr = c / CPR, ch = c % CPR;
    const bool valid = rr < R;
    const int gh = valid ? rr / a.W : 0, i = valid ? rr % a.W : 0;
    const __nv_bfloat16 *src =
        q + (static_cast<size_t>(b) * a.W + i) * a.n_q_heads * D + (h * G + gh) * D + ch * 8;
    cp_async16(smem_u32(sQ + rr * RS + ch * 8), src, valid);
  }
  auto load_kv = [&](int buf, int k0) {
    for (int c = tid; c < kAttKeys * CPR; c += 128) {
      const int kr = c / CPR, ch = c % CPR;
      const int k = k0 + kr;
      const bool valid = k < g.k_end;
      const __nv_bfloat16 *sk = ring_k, *sv = ring_v;
      size_t off = 0;
      if (valid) {
        if (k < g.n_ctx) {
          const long long p = g.p_lo + k;
          off = ((static_cast<size_t>(b) * a.n_kv_heads + h) * a.cap + p % a.cap) * D;
        } else {
          sk = blk_k;
          sv = blk_v;
          off = ((static_cast<size_t>(b) * a.n_kv_heads + h) * a.W + (k - g.n_ctx)) * D;
        }
      }
      cp_async16(smem_u32(sK + (buf * kAttKeys + kr) * RS + ch * 8), sk + off + ch * 8, valid);
      cp_async16(smem_u32(sV + (buf * kAttKeys + kr) * RS + ch * 8), sv + off + ch * 8, valid);
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

  int n_blocks = g.k_end > g.k_begin ? (g.k_end - g.k_begin + kAttKeys - 1) / kAttKeys : 0;
  if (n_blocks > 0) load_kv(0, g.k_begin);
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();

  // Q fragments (A operand), kept in registers for the whole key range
  uint32_t qf[D / 16][4];
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const int mi = lane >> 3;
    const int row = warp * 16 + (mi & 1) * 8 + (lane & 7);
    const int col = ks * 16 + (mi >> 1) * 8;
    ldsm_x4(smem_u32(sQ + row * RS + col), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
  }

  for (int blk = 0; blk < n_blocks; ++blk) {
    const int buf = blk & 1;
    const int k0 = g.k_begin + blk * kAttKeys;
    if (blk + 1 < n_blocks) load_kv(buf ^ 1, k0 + kAttKeys);
    cp_async_commit();

    // S = Q K^T for 16 rows x 64 keys
    float s[kAttKeys / 8][4];
#pragma unroll
    for (int nt = 0; nt < kAttKeys / 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int nt = 0; nt < kAttKeys / 8; nt += 2) {
        const int mi = lane >> 3;
        const int key = (nt + (mi >> 1)) * 8 + (lane & 7);
        const int col = ks * 16 + (mi & 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_u32(sK + (buf * kAttKeys + key) * RS + col), b0, b1, b2, b3);
        mma16816(s[nt], qf[ks], b0, b1);
        mma16816(s[nt + 1], qf[ks], b2, b3);
      }
    }
    // mask + online softmax (base 2)
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < kAttKeys / 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int k = k0 + nt * 8 + 2 * t4 + (e & 1);
        const bool top = e < 2;
        const bool vis = (top ? rvA : rvB) && att_visible(a, g, top ? iA : iB, k);
        s[nt][e] = vis ? s[nt][e] * sl2 : -INFINITY;
        mx[top ? 0 : 1] = fmaxf(mx[top ? 0 : 1], s[nt][e]);
      }
    }
    float alpha[2];
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
    for (int nt = 0; nt < kAttKeys / 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hr = e < 2 ? 0 : 1;
        const float pv = (s[nt][e] == -INFINITY) ? 0.f : exp2f(s[nt][e] - m_run[hr]);
        s[nt][e] = pv;
        ls[hr] += pv;
      }
    }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      ls[hr] += __shfl_xor_sync(0xffffffffu, ls[hr], 1);
      ls[hr] += __shfl_xor_sync(0xffffffffu, ls[hr], 2);
      l_run[hr] = l_run[hr] * alpha[hr] + ls[hr];
    }
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      o[n][0] *= alpha[0];
      o[n][1] *= alpha[0];
      o[n][2] *= alpha[1];
      o[n][3] *= alpha[1];
    }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < kAttKeys / 16; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int nd = 0; nd < D / 8; nd += 2) {
        const int mi = lane >> 3;
        const int key = kk * 16 + (mi & 1) * 8 + (lane & 7);
        const int col = (nd + (mi >> 1)) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_u32(sV + (buf * kAttKeys + key) * RS + col), b0, b1, b2, b3);
        mma16816(o[nd], pa, b0, b1);
        mma16816(o[nd + 1], pa, b2, b3);
      }
    }
    cp_async_wait<0>();
    __syncthreads();
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
}

// Merge the splits: out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.  One warp per
// query row; lanes own D/32 consecutive output dims and the split weights are computed
// by lanes and broadcast, so the per-split loads are independent of each other.
template <typename T, int D>
__global__ void __launch_bounds__(256) attention_combine_kernel(AttArgs a) {
  const int bh = blockIdx.x;
  const int b = bh / a.n_kv_heads, h = bh % a.n_kv_heads;
  const int G = a.n_q_heads / a.n_kv_heads;
  const int R = G * a.W;
  const int rr = blockIdx.y * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  if (rr >= R) return;
  constexpr int PER = D / 32;
  const float *po = a.part_o + static_cast<size_t>(bh) * a.n_splits * kAttRows * D;
  const float2 *pml = a.part_ml + static_cast<size_t>(bh) * a.n_splits * kAttRows;
  float M = -INFINITY;
  for (int s = lane; s < a.n_splits; s += 32) {
    const float2 ml = pml[s * kAttRows + rr];
    if (ml.y > 0.f) M = fmaxf(M, ml.x);
  }
  M = warp_max(M);
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float L = 0.f;
  for (int s0 = 0; s0 < a.n_splits; s0 += 32) {
    const int s = s0 + lane;
    float wgt = 0.f;
    if (s < a.n_splits) {
      const float2 ml = pml[s * kAttRows + rr];
      if (ml.y > 0.f) {
        wgt = exp2f(ml.x - M);
        L += wgt * ml.y;
      }
    }
    const int cnt = min(32, a.n_splits - s0);
#pragma unroll 4
    for (int j = 0; j < cnt; ++j) {
      const float wj = __shfl_sync(0xffffffffu, wgt, j);
      const float *os = po + (static_cast<size_t>(s0 + j) * kAttRows + rr) * D + lane * PER;
      if (PER == 4) {
        const float4 o = *reinterpret_cast<const float4 *>(os);
        acc[0] += wj * o.x;
        acc[1] += wj * o.y;
        acc[2] += wj * o.z;
        acc[3] += wj * o.w;
      } else {
        const float2 o = *reinterpret_cast<const float2 *>(os);
        acc[0] += wj * o.x;
        acc[1] += wj * o.y;
      }
    }
  }
  L = warp_sum(L);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const int gh = rr / a.W, i = rr % a.W;
  T *out = static_cast<T *>(a.out) +
           (static_cast<size_t>(b) * a.W + i) * a.n_q_heads * D + (h * G + gh) * D + lane * PER;
#pragma unroll
  for (int e = 0; e < PER; ++e) out[e] = from_f<T>(acc[e] * inv);
}

// fp32 path (small geometries): one CTA per (query head, request), exact fp32 softmax.
__global__ void __launch_bounds__(128) attention_f32_kernel(AttArgs a) {
  extern __shared__ float sc[];  // [n_keys_max]
  const int qh = blockIdx.x, b = blockIdx.y;
  const int G = a.n_q_heads / a.n_kv_heads;
  const int h = qh / G;
  const int D = a.head_dim;
  pdl_wait();
  pdl_trigger();
  AttGeom g = att_geom(a, b, 0);
  g.k_begin = 0;
  g.k_end = g.n_keys;
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
    for (int k = threadIdx.x; k < g.n_keys; k += blockDim.x) {
      float sdot = -INFINITY;
      if (att_visible(a, g, i, k)) {
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
    for (int k = threadIdx.x; k < g.n_keys; k += blockDim.x) {
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
      for (int k = 0; k < g.n_keys; ++k)
        if (sc[k] != 0.f) acc += sc[k] * key_ptr(k, true)[d];
      float *out = static_cast<float *>(a.out) +
                   (static_cast<size_t>(b) * a.W + i) * a.n_q_heads * D + qh * D;
      out[d] = acc / L;
    }
    __syncthreads();
  }
}

size_t attention_smem_bytes(int head_dim) {
  return static_cast<size_t>(kAttRows + 4 * kAttKeys) * (head_dim + kAttPad) * 2;
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
  const int R = a.n_q_heads / a.n_kv_heads * a.W;
  if (a.head_dim == 128) {
    static bool set = false;
    if (!set) {
      cudaFuncSetAttribute(attention_bf16_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
      set = true;
    }
    e = launch_pdl(attention_bf16_kernel<128>, dim3(a.n_splits, a.n_kv_heads, a.B), dim3(128),
                   smem, stream, a);
    if (e == cudaSuccess)
      e = launch_pdl(attention_combine_kernel<__nv_bfloat16, 128>, dim3(a.B * a.n_kv_heads, (R + 7) / 8),
                     dim3(256), 0, stream, a);
  } else {
    static bool set = false;
    if (!set) {
      cudaFuncSetAttribute(attention_bf16_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
      set = true;
    }
    e = launch_pdl(attention_bf16_kernel<64>, dim3(a.n_splits, a.n_kv_heads, a.B), dim3(128), smem,
                   stream, a);
    if (e == cudaSuccess)
      e = launch_pdl(attention_combine_kernel<__nv_bfloat16, 64>, dim3(a.B * a.n_kv_heads, (R + 7) / 8),
                     dim3(256), 0, stream, a);
  }
  if (e != cudaSuccess) return std::string("attention launch: ") + cudaGetErrorString(e);
  return {};
}

}  // namespace bd
