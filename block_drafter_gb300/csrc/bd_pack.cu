// Packed weight image: every projection matrix stored as contiguous 16 KB boxes (128 rows
// x 128 bytes of K) in the 128-byte-swizzled order the tensor cores read from shared
// memory, so a GEMM pipeline stage is one contiguous bulk copy of kbox boxes.  In a bf16
// config every matrix but the feature projection W_feature is converted to fp16 on the way
// (exact within fp16's range down to 2^-14); W_feature is a pure permutation (plus zero
// padding of partial tiles).
#include "bd_device.cuh"
#include "bd_internal.h"

#include <string>

namespace bd {

BD_DEFINE_ERROR_TAKER(take_error_word_pack)

PackedLayout packed_layout(const bd_config *c) {
  PackedLayout L = {};
  const int e = c->dtype == BD_BF16 ? 2 : 4;
  const int H = c->hidden, QD = c->n_q_heads * c->head_dim, KD = c->n_kv_heads * c->head_dim;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 1023) / 1024 * 1024;
    return o;
  };
  L.w_feature = take(packed_matrix_bytes(H, c->n_target_layers * H, e, false));
  L.head = take(packed_matrix_bytes(c->vocab, H, e, false));
  if (c->code_width > 0) {
    L.g_recv = take(packed_matrix_bytes(c->msg_width, c->code_width, e, false));
    L.g_pred = take(packed_matrix_bytes(c->msg_width, c->code_width, e, false));
    L.a_val = take(packed_matrix_bytes(c->msg_width, c->code_width, e, false));
  }
  for (int l = 0; l < c->n_layers; ++l) {
    L.wq[l] = take(packed_matrix_bytes(QD, H, e, false));
    L.wk[l] = take(packed_matrix_bytes(KD, H, e, false));
    L.wv[l] = take(packed_matrix_bytes(KD, H, e, false));
    L.wo[l] = take(packed_matrix_bytes(H, QD, e, false));
    L.gate_up[l] = take(packed_matrix_bytes(c->ffn, H, e, true));
    L.w_down[l] = take(packed_matrix_bytes(H, c->ffn, e, false));
    if (c->code_width > 0) {
      L.r_read[l] = take(packed_matrix_bytes(c->code_width, H, e, false));
      L.w_write[l] = take(packed_matrix_bytes(H, c->msg_width, e, false));
    }
    if (c->conv_group > 0) {
      L.conv_a[l] = take(packed_matrix_bytes(4 * H / c->conv_group, H, e, false));
      L.conv_m[l] = take(packed_matrix_bytes(4 * H / c->conv_group, H, e, false));
    }
  }
  L.total = off;
  return L;
}

// bf16 -> fp16 of 8 packed values.  Every bf16 value within fp16's finite range converts
// exactly except those below 2^-14, whose fp16 subnormal keeps an absolute precision of
// 2^-25; a value beyond +-65504 sets the range error.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
    bad |= fabsf(f.x) > 65504.f || fabsf(f.y) > 65504.f;
    const __half2 h = __floats2half2_rn(f.x, f.y);
    w[i] = *reinterpret_cast<const uint32_t *>(&h);
  }
  if (bad) atomicOr(&g_error_word, DEVERR_RANGE);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// One CTA per 16 KB box.  Pair images take rows 0..63 of each tile from src0 and rows
// 64..127 from src1 (the same feature rows).  to_f16: bf16 source values stored as fp16.
__global__ void __launch_bounds__(256) pack_kernel(const uint8_t *src0, const uint8_t *src1,
                                                   int rows, int row_bytes, int pair, int n_kb,
                                                   int to_f16, uint8_t *dst) {
  pdl_wait();
  pdl_trigger();
  const size_t box = blockIdx.x;
  const int rt = static_cast<int>(box / n_kb), kbx = static_cast<int>(box % n_kb);
  uint8_t *out = dst + box * kPackBox;
  for (int q = threadIdx.x; q < 1024; q += blockDim.x) {
    const int r = q >> 3, c = q & 7;
    const uint8_t *src = src0;
    int row = rt * 128 + r;
    if (pair) {
      row = rt * 64 + (r & 63);
      src = r < 64 ? src0 : src1;
    }
    const int col = kbx * 128 + c * 16;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (row < rows && col < row_bytes) {
      v = *reinterpret_cast<const uint4 *>(src + static_cast<size_t>(row) * row_bytes + col);
      if (to_f16) v = bf16x8_to_f16x8(v);
    }
    *reinterpret_cast<uint4 *>(out + r * 128 + ((c ^ (r & 7)) << 4)) = v;
  }
}

static std::string pack_one(const void *src0, const void *src1, int rows, int K, int elem,
                            bool pair, void *dst, cudaStream_t s, bool to_f16 = false) {
  const int n_kb = static_cast<int>(packed_kb(K, elem));
  const size_t rt = pair ? (static_cast<size_t>(rows) + 63) / 64 : (static_cast<size_t>(rows) + 127) / 128;
  const size_t boxes = rt * n_kb;
  if (boxes == 0) return {};
  if (boxes > 0x7fffffffull) return "matrix too large to pack";
  cudaError_t e = launch_pdl(pack_kernel, dim3(static_cast<unsigned>(boxes)), dim3(256), 0, s,
                             static_cast<const uint8_t *>(src0), static_cast<const uint8_t *>(src1),
                             rows, K * elem, pair ? 1 : 0, n_kb, to_f16 ? 1 : 0,
                             static_cast<uint8_t *>(dst));
  return e == cudaSuccess ? std::string() : std::string("pack: ") + cudaGetErrorString(e);
}

std::string pack_all(const bd_config *c, const bd_weights *w, uint8_t *base, cudaStream_t s) {
  const PackedLayout L = packed_layout(c);
  const int e = c->dtype == BD_BF16 ? 2 : 4;
  const int H = c->hidden, QD = c->n_q_heads * c->head_dim, KD = c->n_kv_heads * c->head_dim;
  std::string err;
#define BD_PACK(src0, src1, rows, K, pair, off)                                   \
  if ((err = pack_one(src0, src1, rows, K, e, pair, base + (off), s)).size()) return err;
  // matrices whose products take fp16 operands in a bf16 config (packed_f16())
#define BD_PACK16(src0, src1, rows, K, pair, off)                                              \
  if ((err = pack_one(src0, src1, rows, K, e, pair, base + (off), s, f16)).size()) return err;
  const bool f16 = packed_f16(c);
  BD_PACK(w->w_feature, nullptr, H, c->n_target_layers * H, false, L.w_feature);
  BD_PACK16(w->embed_head, nullptr, c->vocab, H, false, L.head);
  if (c->code_width > 0) {
    BD_PACK16(w->g_recv, nullptr, c->msg_width, c->code_width, false, L.g_recv);
    BD_PACK16(w->g_pred, nullptr, c->msg_width, c->code_width, false, L.g_pred);
    BD_PACK16(w->a_val, nullptr, c->msg_width, c->code_width, false, L.a_val);
  }
  for (int l = 0; l < c->n_layers; ++l) {
    const bd_layer_weights &W = w->layer[l];
    BD_PACK16(W.wq, nullptr, QD, H, false, L.wq[l]);
    BD_PACK16(W.wk, nullptr, KD, H, false, L.wk[l]);
    BD_PACK16(W.wv, nullptr, KD, H, false, L.wv[l]);
    BD_PACK16(W.wo, nullptr, H, QD, false, L.wo[l]);
    BD_PACK16(W.w_gate, W.w_up, c->ffn, H, true, L.gate_up[l]);
    BD_PACK16(W.w_down, nullptr, H, c->ffn, false, L.w_down[l]);
    if (c->code_width > 0) {
      BD_PACK16(W.r_read, nullptr, c->code_width, H, false, L.r_read[l]);
      BD_PACK16(W.w_write, nullptr, H, c->msg_width, false, L.w_write[l]);
    }
    if (c->conv_group > 0) {
      BD_PACK16(W.conv_delta_a, nullptr, 4 * H / c->conv_group, H, false, L.conv_a[l]);
      BD_PACK16(W.conv_delta_m, nullptr, 4 * H / c->conv_group, H, false, L.conv_m[l]);
    }
  }
#undef BD_PACK
#undef BD_PACK16
  return {};
}

}  // namespace bd
