// mxattn_attention_noalloc: the whole MXAttention forward for callers that
// cannot allocate device memory.
//
// Some callers have no way to allocate: a plugin interface of a host framework
// that hands an op only its input and output tensors, a process whose device
// memory is fully pre-partitioned by another allocator, or a latency-critical
// loop that must not call cudaMalloc (which can synchronize the device).
// mxattn_attention needs intermediate buffers for the quantized Q, K and V;
// this entry point keeps them in one file-scope device array instead, so the
// caller only passes the bf16 inputs and the fp32 output.
//
// The array is static device memory of the library module: every GPU on which
// the library is used holds kScratchBytes of it until the process exits.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/mxattn.h"
#include "internal.h"

namespace mxattn {

// Maximum scratch: 32 MiB (quantized Q, K, V codes and their scale atoms).
constexpr size_t kScratchBytes = size_t(32) << 20;

namespace {

__device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

// Device address of g_noalloc_scratch on the current device. In host code the
// symbol is only a host-side stand-in, so the address is looked up once per
// device (with that device current) and cached. The cached address is valid
// for the life of the device's primary context: after cudaDeviceReset the
// module is loaded again, possibly elsewhere, so a process that resets a
// device must not call this entry point on it again.
uint8_t* scratch_on_current_device(cudaError_t* err) {
  static uint8_t* addr[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = static_cast<uint8_t*>(p);
  }
  return addr[dev];
}

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// q, k, v and out must be device memory of the current device: the kernels run
// there and would otherwise read another GPU's memory without peer access.
bool on_current_device(const void* p, int dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // clear the (non-sticky) error left by an unknown pointer
    return false;
  }
  return (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) && a.device == dev;
}

}  // namespace

size_t noalloc_scratch_needed(int64_t B, int64_t H, int64_t N) {
  return 2 * up256(mxattn_qk_codes_bytes(B, H, N)) + 2 * up256(mxattn_qk_scales_bytes(B, H, N)) +
         up256(mxattn_v_codes_bytes(B, H, N)) + up256(mxattn_v_scales_bytes(B, H, N));
}

}  // namespace mxattn

using namespace mxattn;

extern "C" size_t mxattn_attention_noalloc_max_scratch_bytes(void) { return kScratchBytes; }

extern "C" mxattn_status mxattn_attention_noalloc(const void* q, const void* k, const void* v, int64_t B, int64_t H,
                                                  int64_t N, int64_t D, int causal, float* out, void* stream) {
  if (B < 0 || H < 0 || N < 0) {
    set_last_error("mxattn_attention_noalloc: negative size");
    return MXATTN_ERR_INVALID_ARG;
  }
  if (D != kD) {
    set_last_error("mxattn_attention_noalloc: head dimension must be 128");
    return MXATTN_ERR_UNSUPPORTED;
  }
  if (B == 0 || H == 0 || N == 0) return MXATTN_OK;
  // the same bounds as every other entry point, before any size product is formed
  if (B > 65535 || H > 65535 || B * H > 65535 || N >= (int64_t(1) << 31) - kTile) {
    set_last_error("mxattn_attention_noalloc: B*H must be at most 65535 and N below 2^31 - 128");
    return MXATTN_ERR_UNSUPPORTED;
  }
  const size_t need = noalloc_scratch_needed(B, H, N);
  if (need > kScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "mxattn_attention_noalloc: B*H*N = %lld needs %zu scratch bytes, more than the fixed %zu; "
             "use mxattn_attention_host or the separate entry points with caller buffers",
             (long long)(B * H * N), need, kScratchBytes);
    set_last_error(msg);
    return MXATTN_ERR_UNSUPPORTED;
  }
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr) {
    set_last_error("mxattn_attention_noalloc: q, k, v and out must be non-NULL");
    return MXATTN_ERR_INVALID_ARG;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || !on_current_device(q, dev) || !on_current_device(k, dev) ||
      !on_current_device(v, dev) || !on_current_device(out, dev)) {
    set_last_error("mxattn_attention_noalloc: q, k, v and out must be device memory of the current device");
    return MXATTN_ERR_INVALID_ARG;
  }
  cudaError_t e = cudaSuccess;
  uint8_t* s = scratch_on_current_device(&e);
  if (s == nullptr) {
    char msg[256];
    snprintf(msg, sizeof msg, "mxattn_attention_noalloc: scratch address lookup failed: %s", cudaGetErrorString(e));
    set_last_error(msg);
    return MXATTN_ERR_CUDA;
  }
  uint8_t* qc = s;
  uint8_t* kc = qc + up256(mxattn_qk_codes_bytes(B, H, N));
  uint8_t* qs = kc + up256(mxattn_qk_codes_bytes(B, H, N));
  uint8_t* ks = qs + up256(mxattn_qk_scales_bytes(B, H, N));
  uint8_t* vc = ks + up256(mxattn_qk_scales_bytes(B, H, N));
  uint8_t* vs = vc + up256(mxattn_v_codes_bytes(B, H, N));
  // Every byte the forward reads is rewritten by the quantizers below, so
  // nothing in the scratch needs clearing between calls.
  const mxattn_status st = mxattn_quantize_qkv(q, k, v, B, H, N, D, qc, qs, kc, ks, vc, vs, stream);
  if (st != MXATTN_OK) return st;
  return mxattn_forward(qc, qs, kc, ks, vc, vs, v, B, H, N, D, causal, out, stream);
}
