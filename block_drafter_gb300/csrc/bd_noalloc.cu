// LM-head argmax for callers that cannot allocate device memory.
//
// Some callers hold no device allocator of their own: a serving engine whose memory
// pool owns every device byte after start-up, or a host program that embeds this library
// through a plugin interface without an allocation hook.  They cannot provide the
// workspace bd_lm_head_argmax needs.  This variant takes its scratch from one file-scope
// device array instead, so a call needs only its inputs and outputs.
//
// The array is part of the library's device image: every GPU that loads the library
// holds it until the process exits.  All calls share it and it keeps the last call's
// contents, so calls that overlap on the GPU (two streams, or two threads) race; the
// counters that must start at zero are cleared by each call before its kernels run.
// The host needs the array's device address, which cudaGetSymbolAddress provides; the
// first call on a device looks it up (with that device current) and caches it, so that
// first call should come before any stream capture.  The cached address belongs to the
// device's context of that moment: after cudaDeviceReset on that device this entry point
// must not be called again in the same process.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "bd_internal.h"
#include "bd_kernels.h"
#include "blockdrafter.h"

namespace bd {
namespace {

// Scratch layout (bytes, each region 256-aligned):
//   split hidden rows  2 * 32 * 8192 * 2            =  1 MiB
//   per-tile maxima    2048 * 32 * 4 (+ indices)    =  0.5 MiB
//   tile counters      2 * 2048 * 4                 = 16 KiB
//   stream-K partials  160 * 2 * 64 * 128 * 4       = 10 MiB
constexpr size_t kMaxRows = BD_NOALLOC_MAX_ROWS;
constexpr size_t kMaxHidden = BD_NOALLOC_MAX_HIDDEN;
constexpr size_t kMaxTiles = BD_NOALLOC_MAX_VOCAB / 128;
constexpr size_t kMaxCtas = 160;
constexpr size_t kSplitBytes = 2 * kMaxRows * kMaxHidden * 2;
constexpr size_t kAmaxBytes = kMaxTiles * kMaxRows * 4;
constexpr size_t kCounterBytes = 2 * kMaxTiles * 4;
constexpr size_t kPartialFloats = kMaxCtas * 2 * (2 * kMaxRows) * kBM;
constexpr size_t kScratchBytes = kSplitBytes + 2 * kAmaxBytes + kCounterBytes + kPartialFloats * 4;
static_assert(kScratchBytes <= BD_NOALLOC_SCRATCH_BYTES, "scratch layout exceeds the stated size");

static __device__ __align__(256) unsigned char g_head_scratch[BD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char *g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
std::string scratch_address(unsigned char **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return std::string("cudaGetDevice: ") + cudaGetErrorString(e);
  if (dev < 0 || dev >= kMaxDevices) return "device ordinal out of range";
  std::lock_guard<std::mutex> g(g_mu);
  if (!g_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_head_scratch);
    if (e != cudaSuccess) return std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e);
    g_addr[dev] = static_cast<unsigned char *>(p);
  }
  *out = g_addr[dev];
  return {};
}

bd_status fail(bd_status s, const std::string &msg) {
  set_last_error(msg);
  return s;
}

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace
}  // namespace bd

extern "C" bd_status bd_lm_head_argmax_noalloc(const bd_config *cfg, const bd_weights *w,
                                               const float *hidden, int rows, int32_t *token_out,
                                               float *max_logit_out, void *stream_) {
  using namespace bd;
  // the whole configuration is checked as every entry point checks it: the packed image's
  // head offset depends on every layer's sizes
  const std::string bad_cfg = validate_config(cfg);
  if (!bad_cfg.empty()) return fail(BD_ERR_INVALID_ARG, bad_cfg);
  if (rows < 1 || static_cast<size_t>(rows) > kMaxRows || static_cast<size_t>(cfg->hidden) > kMaxHidden ||
      static_cast<size_t>(cfg->vocab) > BD_NOALLOC_MAX_VOCAB) {
    char b[200];
    snprintf(b, sizeof b,
             "no-allocation head supports rows <= %d, hidden <= %d, vocab <= %d (got %d, %d, %d)",
             BD_NOALLOC_MAX_ROWS, BD_NOALLOC_MAX_HIDDEN, BD_NOALLOC_MAX_VOCAB, rows, cfg->hidden,
             cfg->vocab);
    return fail(BD_ERR_INVALID_ARG, b);
  }
  if (!w || !w->embed_head || (reinterpret_cast<uintptr_t>(w->embed_head) & 15u))
    return fail(BD_ERR_INVALID_ARG, "embed_head NULL or misaligned");
  if (!hidden || (reinterpret_cast<uintptr_t>(hidden) & 15u))
    return fail(BD_ERR_INVALID_ARG, "hidden NULL or misaligned");
  if (!token_out) return fail(BD_ERR_INVALID_ARG, "token_out NULL");
  if (static_cast<size_t>(num_sms()) > kMaxCtas)
    return fail(BD_ERR_UNSUPPORTED, "more SMs than the no-allocation scratch was sized for");

  unsigned char *base = nullptr;
  std::string err = scratch_address(&base);
  if (!err.empty()) return fail(BD_ERR_CUDA, err);
  const size_t m_tiles = (static_cast<size_t>(cfg->vocab) + 127) / 128;
  size_t off = 0;
  void *hl = base + off;
  off += up256(kSplitBytes);
  float *amax_val = reinterpret_cast<float *>(base + off);
  off += up256(kAmaxBytes);
  int32_t *amax_idx = reinterpret_cast<int32_t *>(base + off);
  off += up256(kAmaxBytes);
  unsigned *counters = reinterpret_cast<unsigned *>(base + off);
  off += up256(kCounterBytes);
  float *partials = reinterpret_cast<float *>(base + off);

  cudaStream_t s = static_cast<cudaStream_t>(stream_);
  // the first kernel clears the tile counters before the GEMM uses them
  const ZeroSpan zero{counters, 2 * m_tiles};
  // the packed head is fp16 in a bf16 config (fp16 hidden rows); the raw head takes the
  // rows as a bf16 hi/lo pair
  const bool head16 = w->packed != nullptr && packed_f16(cfg);
  const bool split = cfg->dtype == BD_BF16 && !head16;
  const size_t pad = (static_cast<size_t>(rows) + 15) / 16 * 16;
  err = head16  ? launch_rows_f16(hidden, static_cast<size_t>(rows) * cfg->hidden, hl, zero, s)
        : split ? launch_split_rows(hidden, static_cast<size_t>(rows) * cfg->hidden, hl,
                                    pad * cfg->hidden, zero, s)
                : launch_zero(zero, s);
  if (!err.empty()) return fail(BD_ERR_CUDA, err);
  GemmPlan p;
  memset(&p, 0, sizeof p);
  p.dtype = head16 ? GT_F16 : (split ? GT_BF16 : GT_F32);
  p.x = (split || head16) ? static_cast<const void *>(hl) : hidden;
  p.n_tokens = rows;
  p.K = cfg->hidden;
  p.split = split;
  p.w[0].ptr = w->embed_head;
  p.w[0].rows = cfg->vocab;
  p.w[0].packed = w->packed ? static_cast<const uint8_t *>(w->packed) + packed_layout(cfg).head
                            : nullptr;
  p.n_w = 1;
  p.args.vocab = cfg->vocab;
  p.args.epi = EPI_ARGMAX;
  p.args.amax_val = amax_val;
  p.args.amax_idx = amax_idx;
  const GemmScratch sc{partials, kPartialFloats, counters, m_tiles};
  err = launch_gemm(p, sc, s);
  if (!err.empty()) return fail(BD_ERR_CUDA, err);
  err = launch_argmax_reduce(amax_val, amax_idx, static_cast<int>(m_tiles), rows, token_out,
                             max_logit_out, s);
  if (!err.empty()) return fail(BD_ERR_CUDA, err);
  return BD_OK;
}
