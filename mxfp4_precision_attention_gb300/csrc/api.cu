// extern "C" boundary of libmxattn: argument validation, the device status
// word, tensor-map encoding and the host-buffer convenience entry point.
// The declarations and their contracts are in include/mxattn.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/mxattn.h"
#include "internal.h"

namespace mxattn {

__device__ int g_status_word;

namespace {

thread_local char t_err[512] = "";
uint32_t g_debug_flags = 0;

mxattn_status fail(mxattn_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof t_err, fmt, ap);
  va_end(ap);
  return st;
}

mxattn_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MXATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
  uintptr_t lo, hi;
};
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }
Range rng(const void* p, size_t n) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return {a, a + n};
}

// Common shape checks. Returns MXATTN_OK and sets *empty when there is no work.
mxattn_status check_shape(int64_t B, int64_t H, int64_t N, int64_t D, bool* empty) {
  if (B < 0 || H < 0 || N < 0) return fail(MXATTN_ERR_INVALID_ARG, "negative size (B=%lld H=%lld N=%lld)",
                                           (long long)B, (long long)H, (long long)N);
  if (D != kD) return fail(MXATTN_ERR_UNSUPPORTED, "head dimension D=%lld unsupported (only 128)", (long long)D);
  *empty = (B == 0 || H == 0 || N == 0);
  if (*empty) return MXATTN_OK;
  if (B * H > 65535) return fail(MXATTN_ERR_UNSUPPORTED, "B*H=%lld exceeds 65535", (long long)(B * H));
  if (N >= (int64_t(1) << 31) - kTile) return fail(MXATTN_ERR_UNSUPPORTED, "N=%lld too large", (long long)N);
  return MXATTN_OK;
}

mxattn_status check_ptr(const void* p, const char* name) {
  if (p == nullptr) return fail(MXATTN_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned16(p)) return fail(MXATTN_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return MXATTN_OK;
}

size_t qk_codes(int64_t B, int64_t H, int64_t N) { return static_cast<size_t>(B * H * N * 64); }
size_t sf_bytes(int64_t B, int64_t H, int64_t N) {
  return static_cast<size_t>(B * H * ceil_div(N, kTile) * kSfAtomBytes);
}
size_t v_codes(int64_t B, int64_t H, int64_t N) {
  return static_cast<size_t>(B * H * kD * (ceil_div(N, kBlock) * kBlock / 2));
}
size_t bf16_bytes(int64_t B, int64_t H, int64_t N) { return static_cast<size_t>(B * H * N * kD * 2); }
size_t f32_bytes(int64_t B, int64_t H, int64_t N) { return static_cast<size_t>(B * H * N * kD * 4); }

#define MX_TRY(expr)                          \
  do {                                        \
    mxattn_status _st = (expr);               \
    if (_st != MXATTN_OK) return _st;         \
  } while (0)

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

mxattn_status check_rule(int rule, double qmax, const char* what) {
  if (rule < kRuleUOS || rule > kRuleCeilQ)
    return fail(MXATTN_ERR_INVALID_ARG, "%s must be 0 (UOS), 1 (OCP), 2 (TFS) or 3 (ceil with qmax)", what);
  if (rule == kRuleCeilQ && !(qmax > 4.0 && qmax <= 8.0))
    return fail(MXATTN_ERR_INVALID_ARG, "qmax must lie in (4, 8] for the ceil rule");
  return MXATTN_OK;
}

// The quantizers launch through a TMA tensor map and report expired waits in
// the device status word.
mxattn_status check_quantizer_runtime() {
  if (get_encoder() == nullptr) return fail(MXATTN_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  if (device_status_ptr() == nullptr) return fail(MXATTN_ERR_CUDA, "device status word unavailable");
  return MXATTN_OK;
}

mxattn_status forward_impl(const void* qc, const void* qs, const void* kc, const void* ks, const void* vc,
                           const void* vs, const void* vb, int64_t B, int64_t H, int64_t N, int64_t D, int causal,
                           void* out, uint8_t* pc, uint8_t* ps, void* stream, int p_rule = kRuleUOS,
                           int placement = kPlacePNQ, double p_qmax = 7.25, const float* q_amax = nullptr,
                           const float* k_amax = nullptr, const float* v_amax = nullptr, bool out_bf16 = false) {
  bool empty = false;
  MX_TRY(check_shape(B, H, N, D, &empty));
  if (empty) return MXATTN_OK;
  MX_TRY(check_ptr(qc, "q_codes"));
  MX_TRY(check_ptr(qs, "q_scales"));
  MX_TRY(check_ptr(kc, "k_codes"));
  MX_TRY(check_ptr(ks, "k_scales"));
  MX_TRY(check_ptr(vc, "v_codes"));
  MX_TRY(check_ptr(vs, "v_scales"));
  MX_TRY(check_ptr(out, "out"));
  if (causal < 0 || causal > 2) return fail(MXATTN_ERR_INVALID_ARG, "causal must be 0, 1 or 2");
  MX_TRY(check_rule(p_rule, p_qmax, "p_rule"));
  if (placement != kPlacePNQ && placement != kPlaceDirect)
    return fail(MXATTN_ERR_INVALID_ARG, "placement must be 0 (PNQ) or 1 (direct)");
  if (causal) MX_TRY(check_ptr(vb, "v_bf16 (required when causal)"));
  if ((pc == nullptr) != (ps == nullptr)) return fail(MXATTN_ERR_INVALID_ARG, "phat dump needs both buffers");
  if (pc) {
    MX_TRY(check_ptr(pc, "phat_codes"));
    MX_TRY(check_ptr(ps, "phat_scales"));
  }
  const bool nv = q_amax != nullptr;
  const size_t sfb = (nv ? 2 : 1) * sf_bytes(B, H, N);
  const Range ro = rng(out, out_bf16 ? bf16_bytes(B, H, N) : f32_bytes(B, H, N));
  const Range ins[] = {rng(qc, qk_codes(B, H, N)), rng(qs, sfb), rng(kc, qk_codes(B, H, N)),
                       rng(ks, sfb),  rng(vc, v_codes(B, H, N)), rng(vs, sfb)};
  for (const Range& r : ins)
    if (overlap(ro, r)) return fail(MXATTN_ERR_INVALID_ARG, "out overlaps an input buffer");
  if (nv) {
    for (const float* am : {q_amax, k_amax, v_amax}) {
      if (am == nullptr || (reinterpret_cast<uintptr_t>(am) & 3u))
        return fail(MXATTN_ERR_INVALID_ARG, "q_amax, k_amax and v_amax must be non-NULL, 4-byte aligned");
      if (overlap(ro, rng(am, sizeof(float)))) return fail(MXATTN_ERR_INVALID_ARG, "out overlaps an amax");
    }
    if (causal == 2) return fail(MXATTN_ERR_INVALID_ARG, "the NVFP4 forward takes causal 0 or 1");
  }
  if (causal && overlap(ro, rng(vb, bf16_bytes(B, H, N))))
    return fail(MXATTN_ERR_INVALID_ARG, "out overlaps v_bf16");
  Mxfp4FwdArgs a;
  a.q_codes = qc;
  a.q_scales = qs;
  a.k_codes = kc;
  a.k_scales = ks;
  a.v_codes = vc;
  a.v_scales = vs;
  a.v_bf16 = vb;
  a.BH = B * H;
  a.N = N;
  a.causal = causal;
  a.out = out_bf16 ? nullptr : static_cast<float*>(out);
  a.out_bf16 = out_bf16 ? out : nullptr;
  a.phat_codes = pc;
  a.phat_scales = ps;
  a.debug_flags = g_debug_flags;
  a.p_rule = p_rule;
  a.placement = placement;
  a.p_qmax = p_qmax;
  a.q_amax = q_amax;
  a.k_amax = k_amax;
  a.v_amax = v_amax;
  if (get_encoder() == nullptr) return fail(MXATTN_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  if (device_status_ptr() == nullptr) return fail(MXATTN_ERR_CUDA, "device status word unavailable");
  cudaError_t e = launch_mxfp4_forward(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mxfp4 forward launch");
  return MXATTN_OK;
}

// Internal copy streams and events of mxattn_attention_host, created once per
// device and reused; a call holds the device's lock while it enqueues and
// waits, so concurrent host calls on one device run one after the other.
constexpr int64_t kHostChunks = 64;  // at most this many chunks (events per direction)
// Input bytes (bf16 Q, K and V) per middle chunk. Smaller chunks add per-chunk
// launch and synchronisation gaps; larger ones lengthen the pipeline's fill
// and drain. Measured best at 50-57 MB on GB300 for both the Wan-shaped
// (compute-bound) and the causal 8192-token (copy-bound) workloads.
constexpr size_t kHostChunkBytes = size_t(52) << 20;
struct HostPipe {
  std::mutex mu;
  cudaStream_t h2d = nullptr, d2h = nullptr, alt = nullptr;
  cudaEvent_t ev_start = nullptr, ev_done = nullptr;
  cudaEvent_t ev_in[kHostChunks] = {}, ev_out[kHostChunks] = {};
  bool ready = false;
};

HostPipe* host_pipe_for_current_device(cudaError_t* err) {
  static HostPipe pipes[64];
  static std::mutex mu;
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  HostPipe& p = pipes[dev];
  if (!p.ready) {
    if ((*err = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking)) != cudaSuccess) return nullptr;
    if ((*err = cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking)) != cudaSuccess) return nullptr;
    if ((*err = cudaStreamCreateWithFlags(&p.alt, cudaStreamNonBlocking)) != cudaSuccess) return nullptr;
    const unsigned fl = cudaEventDisableTiming;
    if ((*err = cudaEventCreateWithFlags(&p.ev_start, fl)) != cudaSuccess) return nullptr;
    if ((*err = cudaEventCreateWithFlags(&p.ev_done, fl)) != cudaSuccess) return nullptr;
    for (int i = 0; i < kHostChunks; i++) {
      if ((*err = cudaEventCreateWithFlags(&p.ev_in[i], fl)) != cudaSuccess) return nullptr;
      if ((*err = cudaEventCreateWithFlags(&p.ev_out[i], fl)) != cudaSuccess) return nullptr;
    }
    p.ready = true;
  }
  return &p;
}

}  // namespace

void set_last_error(const char* msg) { snprintf(t_err, sizeof t_err, "%s", msg); }

int* device_status_ptr() {
  static int* ptrs[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

cudaError_t read_and_clear_device_status(int* status, cudaStream_t s) {
  int* d = device_status_ptr();
  if (d == nullptr) return cudaErrorInvalidDevice;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  e = cudaMemcpy(status, d, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return e;
  return cudaMemset(d, 0, sizeof(int));
}

bool encode_tensor_map(void* map, int dtype_is_bf16, int rank, void* base, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box, int swizzle_bytes) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encoder();
  if (enc == nullptr) return false;
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; i++) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i < rank - 1; i++) gs[i] = strides_bytes[i];
  const CUtensorMapSwizzle sw = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                      : CU_TENSOR_MAP_SWIZZLE_NONE;
  const CUresult r = enc(static_cast<CUtensorMap*>(map),
                         dtype_is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                         static_cast<cuuint32_t>(rank), base, gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace mxattn

using namespace mxattn;

extern "C" {

size_t mxattn_nvfp4_scales_bytes(int64_t B, int64_t H, int64_t N) {
  return B < 0 || H < 0 || N < 0 ? 0 : 2 * sf_bytes(B, H, N);
}
size_t mxattn_qk_codes_bytes(int64_t B, int64_t H, int64_t N) { return B < 0 || H < 0 || N < 0 ? 0 : qk_codes(B, H, N); }
size_t mxattn_qk_scales_bytes(int64_t B, int64_t H, int64_t N) { return B < 0 || H < 0 || N < 0 ? 0 : sf_bytes(B, H, N); }
size_t mxattn_v_codes_bytes(int64_t B, int64_t H, int64_t N) { return B < 0 || H < 0 || N < 0 ? 0 : v_codes(B, H, N); }
size_t mxattn_v_scales_bytes(int64_t B, int64_t H, int64_t N) { return B < 0 || H < 0 || N < 0 ? 0 : sf_bytes(B, H, N); }

mxattn_status mxattn_rotate_quantize_qk(const void* x, int64_t B, int64_t H, int64_t N, int64_t D, void* codes,
                                        void* scales, void* stream) {
  return mxattn_quantize_qk_ex(x, B, H, N, D, MXATTN_RULE_UOS, 7.25, 1, codes, scales, stream);
}

mxattn_status mxattn_quantize_qk_ex(const void* x, int64_t B, int64_t H, int64_t N, int64_t D, int rule,
                                    double qmax, int rotate, void* codes, void* scales, void* stream) {
  t_err[0] = '\0';
  MX_TRY(check_rule(rule, qmax, "rule"));
  if (rotate != 0 && rotate != 1) return fail(MXATTN_ERR_INVALID_ARG, "rotate must be 0 or 1");
  bool empty = false;
  MX_TRY(check_shape(B, H, N, D, &empty));
  if (empty) return MXATTN_OK;
  MX_TRY(check_ptr(x, "x"));
  MX_TRY(check_ptr(codes, "codes"));
  MX_TRY(check_ptr(scales, "scales"));
  const Range rx = rng(x, bf16_bytes(B, H, N)), rc = rng(codes, qk_codes(B, H, N)), rs = rng(scales, sf_bytes(B, H, N));
  if (overlap(rx, rc) || overlap(rx, rs) || overlap(rc, rs))
    return fail(MXATTN_ERR_INVALID_ARG, "x, codes and scales must not overlap");
  MX_TRY(check_quantizer_runtime());
  cudaError_t e =
      launch_rotate_quantize_qk(x, B * H, N, codes, scales, rule, qmax, rotate, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rotate_quantize_qk launch");
  return MXATTN_OK;
}

mxattn_status mxattn_quantize_v(const void* v, int64_t B, int64_t H, int64_t N, int64_t D, void* codes,
                                void* scales, void* stream) {
  return mxattn_quantize_v_ex(v, B, H, N, D, MXATTN_RULE_UOS, 7.25, codes, scales, stream);
}

mxattn_status mxattn_quantize_v_ex(const void* v, int64_t B, int64_t H, int64_t N, int64_t D, int rule, double qmax,
                                   void* codes, void* scales, void* stream) {
  t_err[0] = '\0';
  MX_TRY(check_rule(rule, qmax, "rule"));
  bool empty = false;
  MX_TRY(check_shape(B, H, N, D, &empty));
  if (empty) return MXATTN_OK;
  MX_TRY(check_ptr(v, "v"));
  MX_TRY(check_ptr(codes, "codes"));
  MX_TRY(check_ptr(scales, "scales"));
  const Range rv = rng(v, bf16_bytes(B, H, N)), rc = rng(codes, v_codes(B, H, N)), rs = rng(scales, sf_bytes(B, H, N));
  if (overlap(rv, rc) || overlap(rv, rs) || overlap(rc, rs))
    return fail(MXATTN_ERR_INVALID_ARG, "v, codes and scales must not overlap");
  MX_TRY(check_quantizer_runtime());
  cudaError_t e = launch_quantize_v(v, B * H, N, codes, scales, rule, qmax, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantize_v launch");
  return MXATTN_OK;
}

static mxattn_status nvfp4_quantize(const void* x, int64_t B, int64_t H, int64_t N, int64_t D, void* codes,
                                    void* scales, float* amax, void* stream, int is_v) {
  t_err[0] = '\0';
  bool empty = false;
  MX_TRY(check_shape(B, H, N, D, &empty));
  if (empty) return MXATTN_OK;
  MX_TRY(check_ptr(x, "x"));
  MX_TRY(check_ptr(codes, "codes"));
  MX_TRY(check_ptr(scales, "scales"));
  if (amax == nullptr || (reinterpret_cast<uintptr_t>(amax) & 3u))
    return fail(MXATTN_ERR_INVALID_ARG, "amax must be a non-NULL, 4-byte aligned device float");
  const size_t nc = is_v ? v_codes(B, H, N) : qk_codes(B, H, N);
  const Range rx = rng(x, bf16_bytes(B, H, N)), rc = rng(codes, nc), rs = rng(scales, 2 * sf_bytes(B, H, N)),
              ra = rng(amax, sizeof(float));
  if (overlap(rx, rc) || overlap(rx, rs) || overlap(rc, rs) || overlap(ra, rx) || overlap(ra, rc) || overlap(ra, rs))
    return fail(MXATTN_ERR_INVALID_ARG, "x, codes, scales and amax must not overlap");
  MX_TRY(check_quantizer_runtime());
  const QuantizeJob j{x, codes, scales, kRuleUOS, 7.25, is_v, 0, amax};
  cudaError_t e = launch_quantize(&j, 1, B * H, N, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "nvfp4 quantizer launch");
  return MXATTN_OK;
}

mxattn_status mxattn_nvfp4_quantize_qk(const void* x, int64_t B, int64_t H, int64_t N, int64_t D, void* codes,
                                       void* scales, float* amax, void* stream) {
  return nvfp4_quantize(x, B, H, N, D, codes, scales, amax, stream, 0);
}

mxattn_status mxattn_nvfp4_quantize_v(const void* v, int64_t B, int64_t H, int64_t N, int64_t D, void* codes,
                                      void* scales, float* amax, void* stream) {
  return nvfp4_quantize(v, B, H, N, D, codes, scales, amax, stream, 1);
}

mxattn_status mxattn_quantize_qkv(const void* q, const void* k, const void* v, int64_t B, int64_t H, int64_t N,
                                  int64_t D, void* q_codes, void* q_scales, void* k_codes, void* k_scales,
                                  void* v_codes, void* v_scales, void* stream) {
  t_err[0] = '\0';
  bool empty = false;
  MX_TRY(check_shape(B, H, N, D, &empty));
  if (empty) return MXATTN_OK;
  MX_TRY(check_ptr(q, "q"));
  MX_TRY(check_ptr(k, "k"));
  MX_TRY(check_ptr(v, "v"));
  MX_TRY(check_ptr(q_codes, "q_codes"));
  MX_TRY(check_ptr(q_scales, "q_scales"));
  MX_TRY(check_ptr(k_codes, "k_codes"));
  MX_TRY(check_ptr(k_scales, "k_scales"));
  MX_TRY(check_ptr(v_codes, "v_codes"));
  MX_TRY(check_ptr(v_scales, "v_scales"));
  const size_t xb = bf16_bytes(B, H, N);
  const Range in[3] = {rng(q, xb), rng(k, xb), rng(v, xb)};
  const Range outs[6] = {rng(q_codes, qk_codes(B, H, N)), rng(q_scales, sf_bytes(B, H, N)),
                         rng(k_codes, qk_codes(B, H, N)), rng(k_scales, sf_bytes(B, H, N)),
                         rng(v_codes, mxattn_v_codes_bytes(B, H, N)), rng(v_scales, sf_bytes(B, H, N))};
  for (int i = 0; i < 6; i++) {
    for (int j = 0; j < 3; j++)
      if (overlap(outs[i], in[j])) return fail(MXATTN_ERR_INVALID_ARG, "an output overlaps an input");
    for (int j = i + 1; j < 6; j++)
      if (overlap(outs[i], outs[j])) return fail(MXATTN_ERR_INVALID_ARG, "two outputs overlap");
  }
  MX_TRY(check_quantizer_runtime());
  const QuantizeJob jobs[3] = {{q, q_codes, q_scales, kRuleUOS, 7.25, 0, 1, nullptr},
                               {k, k_codes, k_scales, kRuleUOS, 7.25, 0, 1, nullptr},
                               {v, v_codes, v_scales, kRuleUOS, 7.25, 1, 0, nullptr}};
  cudaError_t e = launch_quantize(jobs, 3, B * H, N, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantize_qkv launch");
  return MXATTN_OK;
}

mxattn_status mxattn_forward(const void* q_codes, const void* q_scales, const void* k_codes, const void* k_scales,
                             const void* v_codes, const void* v_scales, const void* v_bf16, int64_t B, int64_t H,
                             int64_t N, int64_t D, int causal, float* out, void* stream) {
  t_err[0] = '\0';
  if (causal != 0 && causal != 1) return fail(MXATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  return forward_impl(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, v_bf16, B, H, N, D, causal, out,
                      nullptr, nullptr, stream);
}

mxattn_status mxattn_forward_out_bf16(const void* q_codes, const void* q_scales, const void* k_codes,
                                      const void* k_scales, const void* v_codes, const void* v_scales,
                                      const void* v_bf16, int64_t B, int64_t H, int64_t N, int64_t D, int causal,
                                      void* out, void* stream) {
  t_err[0] = '\0';
  if (causal != 0 && causal != 1) return fail(MXATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  return forward_impl(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, v_bf16, B, H, N, D, causal, out,
                      nullptr, nullptr, stream, kRuleUOS, kPlacePNQ, 7.25, nullptr, nullptr, nullptr, true);
}

mxattn_status mxattn_forward_dump_phat(const void* q_codes, const void* q_scales, const void* k_codes,
                                       const void* k_scales, const void* v_codes, const void* v_scales,
                                       const void* v_bf16, int64_t B, int64_t H, int64_t N, int64_t D, int causal,
                                       float* out, uint8_t* phat_codes, uint8_t* phat_scales, void* stream) {
  t_err[0] = '\0';
  if (phat_codes == nullptr || phat_scales == nullptr)
    return fail(MXATTN_ERR_INVALID_ARG, "phat_codes and phat_scales are required");
  if (causal != 0 && causal != 1) return fail(MXATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  return forward_impl(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, v_bf16, B, H, N, D, causal, out,
                      phat_codes, phat_scales, stream);
}

mxattn_status mxattn_forward_ex(const void* q_codes, const void* q_scales, const void* k_codes, const void* k_scales,
                                const void* v_codes, const void* v_scales, const void* v_bf16, int64_t B, int64_t H,
                                int64_t N, int64_t D, int causal, int p_rule, double p_qmax, int placement,
                                float* out, void* stream) {
  t_err[0] = '\0';
  return forward_impl(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, v_bf16, B, H, N, D, causal, out,
                      nullptr, nullptr, stream, p_rule, placement, p_qmax);
}

mxattn_status mxattn_nvfp4_forward(const void* q_codes, const void* q_scales, const float* q_amax,
                                   const void* k_codes, const void* k_scales, const float* k_amax,
                                   const void* v_codes, const void* v_scales, const float* v_amax, const void* v_bf16,
                                   int64_t B, int64_t H, int64_t N, int64_t D, int causal, int placement, float* out,
                                   void* stream) {
  t_err[0] = '\0';
  if (q_amax == nullptr) return fail(MXATTN_ERR_INVALID_ARG, "q_amax is NULL");
  return forward_impl(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, v_bf16, B, H, N, D, causal, out,
                      nullptr, nullptr, stream, kRuleUOS, placement, 7.25, q_amax, k_amax, v_amax);
}

mxattn_status mxattn_nvfp4_forward_dump_phat(const void* q_codes, const void* q_scales, const float* q_amax,
                                             const void* k_codes, const void* k_scales, const float* k_amax,
                                             const void* v_codes, const void* v_scales, const float* v_amax,
                                             const void* v_bf16, int64_t B, int64_t H, int64_t N, int64_t D,
                                             int causal, int placement, float* out, uint8_t* phat_codes,
                                             uint8_t* phat_scales, void* stream) {
  t_err[0] = '\0';
  if (q_amax == nullptr) return fail(MXATTN_ERR_INVALID_ARG, "q_amax is NULL");
  if (phat_codes == nullptr || phat_scales == nullptr) return fail(MXATTN_ERR_INVALID_ARG, "phat dump needs both buffers");
  return forward_impl(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, v_bf16, B, H, N, D, causal, out,
                      phat_codes, phat_scales, stream, kRuleUOS, placement, 7.25, q_amax, k_amax, v_amax);
}

mxattn_status mxattn_forward_bf16(const void* q, const void* k, const void* v, int64_t B, int64_t H, int64_t Nq,
                                  int64_t Nk, int64_t D, int causal, float* out, void* stream) {
  t_err[0] = '\0';
  bool empty = false;
  if (Nk < 0) return fail(MXATTN_ERR_INVALID_ARG, "negative size (Nk=%lld)", (long long)Nk);
  MX_TRY(check_shape(B, H, Nq, D, &empty));
  if (empty) return MXATTN_OK;
  bool no_keys = false;
  MX_TRY(check_shape(B, H, Nk, D, &no_keys));
  if (no_keys) return fail(MXATTN_ERR_INVALID_ARG, "Nk=0 with Nq=%lld queries: softmax over no keys", (long long)Nq);
  MX_TRY(check_ptr(q, "q"));
  MX_TRY(check_ptr(k, "k"));
  MX_TRY(check_ptr(v, "v"));
  MX_TRY(check_ptr(out, "out"));
  if (causal != 0 && causal != 1) return fail(MXATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  const Range ro = rng(out, f32_bytes(B, H, Nq));
  if (overlap(ro, rng(q, bf16_bytes(B, H, Nq))) || overlap(ro, rng(k, bf16_bytes(B, H, Nk))) ||
      overlap(ro, rng(v, bf16_bytes(B, H, Nk))))
    return fail(MXATTN_ERR_INVALID_ARG, "out overlaps an input");
  if (get_encoder() == nullptr) return fail(MXATTN_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  if (device_status_ptr() == nullptr) return fail(MXATTN_ERR_CUDA, "device status word unavailable");
  Bf16FwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.BH = B * H;
  a.Nq = Nq;
  a.Nk = Nk;
  a.causal = causal;
  a.out = out;
  a.debug_flags = g_debug_flags;
  cudaError_t e = launch_bf16_forward(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "bf16 forward launch");
  return MXATTN_OK;
}

size_t mxattn_workspace_bytes(int64_t B, int64_t H, int64_t N) {
  if (B < 0 || H < 0 || N < 0) return 0;
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  return 3 * up(bf16_bytes(B, H, N)) + 2 * up(qk_codes(B, H, N)) + 3 * up(sf_bytes(B, H, N)) +
         up(v_codes(B, H, N)) + up(f32_bytes(B, H, N));
}

mxattn_status mxattn_attention_host(const void* q_host, const void* k_host, const void* v_host, int64_t B, int64_t H,
                                    int64_t N, int64_t D, int causal, float* out_host, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  t_err[0] = '\0';
  bool empty = false;
  MX_TRY(check_shape(B, H, N, D, &empty));
  if (empty) return MXATTN_OK;
  if (!q_host || !k_host || !v_host || !out_host) return fail(MXATTN_ERR_INVALID_ARG, "host pointer is NULL");
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(MXATTN_ERR_INVALID_ARG, "workspace must be non-NULL and 256-byte aligned");
  if (workspace_bytes < mxattn_workspace_bytes(B, H, N))
    return fail(MXATTN_ERR_INVALID_ARG, "workspace too small (%zu < %zu)", workspace_bytes,
                mxattn_workspace_bytes(B, H, N));
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  uint8_t* w = static_cast<uint8_t*>(workspace);
  auto take = [&](size_t n) {
    uint8_t* p = w;
    w += up(n);
    return p;
  };
  const size_t xb = bf16_bytes(B, H, N);
  uint8_t *q = take(xb), *k = take(xb), *v = take(xb);
  uint8_t *qc = take(qk_codes(B, H, N)), *kc = take(qk_codes(B, H, N));
  uint8_t *qs = take(sf_bytes(B, H, N)), *ks = take(sf_bytes(B, H, N)), *vs = take(sf_bytes(B, H, N));
  uint8_t* vc = take(v_codes(B, H, N));
  float* out = reinterpret_cast<float*>(take(f32_bytes(B, H, N)));
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // The heads (B*H, contiguous in every layout) are split into up to
  // kHostChunks chunks. Chunk c's inputs are copied in on one internal
  // stream, quantized and attended on the caller's stream (even c) or a
  // second compute stream (odd c), and its output copied out on a third
  // stream: the copies of neighbouring chunks overlap each other and the
  // kernels, and one chunk's CTAs fill the SMs the previous chunk's last
  // wave leaves idle.
  cudaError_t e;
  HostPipe* hp = host_pipe_for_current_device(&e);
  if (hp == nullptr) return cuda_fail(e, "host copy streams");
  std::lock_guard<std::mutex> lock(hp->mu);
  const int64_t BH = B * H;
  const int64_t NT = ceil_div(N, kTile), npad_half = ceil_div(N, kBlock) * kBlock / 2;
  const size_t xh = static_cast<size_t>(N) * kD * 2, oh = static_cast<size_t>(N) * kD * 4;
  // Chunk boundaries: the first and the last chunk hold one head, so the
  // kernels start after a short copy and the final copy out is short; the
  // heads in between go in chunks of about kHostChunkBytes of input.
  int64_t bounds[kHostChunks + 1];
  int64_t nchunks = 0;
  {
    const int64_t edge = BH >= 4 ? 1 : 0;
    const int64_t mid_heads = BH - 2 * edge;
    const size_t head_in = 3 * xh;
    int64_t per = static_cast<int64_t>((kHostChunkBytes + head_in / 2) / head_in);
    if (per < 1) per = 1;
    if (ceil_div(mid_heads, per) > kHostChunks - 2 * edge) per = ceil_div(mid_heads, kHostChunks - 2 * edge);
    bounds[0] = 0;
    if (edge) bounds[++nchunks] = 1;
    for (int64_t h = edge + per; h < BH - edge; h += per) bounds[++nchunks] = h;
    if (edge) bounds[++nchunks] = BH - 1;
    bounds[++nchunks] = BH;
  }
  const size_t qch = static_cast<size_t>(N) * 64, sfh = static_cast<size_t>(NT) * kSfAtomBytes,
               vch = static_cast<size_t>(kD) * npad_half;
  // copies into the workspace may start once earlier work on `stream` is done
  if ((e = cudaEventRecord(hp->ev_start, s)) != cudaSuccess) return cuda_fail(e, "event record");
  if ((e = cudaStreamWaitEvent(hp->h2d, hp->ev_start, 0)) != cudaSuccess) return cuda_fail(e, "stream wait");
  const char* hq = static_cast<const char*>(q_host);
  const char* hk = static_cast<const char*>(k_host);
  const char* hv = static_cast<const char*>(v_host);
  char* ho = reinterpret_cast<char*>(out_host);
  for (int64_t c = 0; c < nchunks; c++) {
    const int64_t h0 = bounds[c], hn = bounds[c + 1] - bounds[c];
    const size_t xo = h0 * xh, xn = hn * xh;
    if ((e = cudaMemcpyAsync(q + xo, hq + xo, xn, cudaMemcpyHostToDevice, hp->h2d)) != cudaSuccess) return cuda_fail(e, "copy q");
    if ((e = cudaMemcpyAsync(k + xo, hk + xo, xn, cudaMemcpyHostToDevice, hp->h2d)) != cudaSuccess) return cuda_fail(e, "copy k");
    if ((e = cudaMemcpyAsync(v + xo, hv + xo, xn, cudaMemcpyHostToDevice, hp->h2d)) != cudaSuccess) return cuda_fail(e, "copy v");
    if ((e = cudaEventRecord(hp->ev_in[c], hp->h2d)) != cudaSuccess) return cuda_fail(e, "event record");
    cudaStream_t cs = (c & 1) ? hp->alt : s;
    void* cstream = static_cast<void*>(cs);
    if ((e = cudaStreamWaitEvent(cs, hp->ev_in[c], 0)) != cudaSuccess) return cuda_fail(e, "stream wait");
    uint8_t *cq = qc + h0 * qch, *ck = kc + h0 * qch, *cv = vc + h0 * vch;
    uint8_t *sq = qs + h0 * sfh, *sk = ks + h0 * sfh, *sv = vs + h0 * sfh;
    MX_TRY(mxattn_quantize_qkv(q + xo, k + xo, v + xo, 1, hn, N, D, cq, sq, ck, sk, cv, sv, cstream));
    float* co = reinterpret_cast<float*>(reinterpret_cast<char*>(out) + h0 * oh);
    MX_TRY(mxattn_forward(cq, sq, ck, sk, cv, sv, v + xo, 1, hn, N, D, causal, co, cstream));
    if ((e = cudaEventRecord(hp->ev_out[c], cs)) != cudaSuccess) return cuda_fail(e, "event record");
    if ((e = cudaStreamWaitEvent(hp->d2h, hp->ev_out[c], 0)) != cudaSuccess) return cuda_fail(e, "stream wait");
    if ((e = cudaMemcpyAsync(ho + h0 * oh, co, hn * oh, cudaMemcpyDeviceToHost, hp->d2h)) != cudaSuccess)
      return cuda_fail(e, "copy out");
  }
  // `stream` is complete once the last output copy has landed (every chunk's
  // kernels, on either compute stream, precede its output copy)
  if ((e = cudaEventRecord(hp->ev_done, hp->d2h)) != cudaSuccess) return cuda_fail(e, "event record");
  if ((e = cudaStreamWaitEvent(s, hp->ev_done, 0)) != cudaSuccess) return cuda_fail(e, "stream wait");
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "stream synchronize");
  return MXATTN_OK;
}

mxattn_status mxattn_mxf4_mma_rate(int64_t iters, int n, float* d_out, double* flops_out, void* stream) {
  t_err[0] = '\0';
  if (iters < 1 || iters > (int64_t(1) << 27))
    return fail(MXATTN_ERR_INVALID_ARG, "iters=%lld outside [1, 2^27]", (long long)iters);
  if (n != 128 && n != 256) return fail(MXATTN_ERR_INVALID_ARG, "n=%d must be 128 or 256", n);
  if (d_out != nullptr && (reinterpret_cast<uintptr_t>(d_out) & 3u) != 0)
    return fail(MXATTN_ERR_INVALID_ARG, "d_out is not 4-byte aligned");
  if (device_status_ptr() == nullptr) return fail(MXATTN_ERR_CUDA, "device status word unavailable");
  int ctas = 0;
  cudaError_t e = launch_mxf4_mma_rate(iters, n, d_out, &ctas, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mma rate probe launch");
  if (flops_out != nullptr) *flops_out = mxf4_mma_rate_flops(iters, n, ctas);
  return MXATTN_OK;
}

mxattn_status mxattn_check(void* stream) {
  int st = 0;
  cudaError_t e = read_and_clear_device_status(&st, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mxattn_check");
  if (st != 0) return fail(MXATTN_ERR_TIMEOUT, "a kernel's bounded wait expired (status %d)", st);
  return MXATTN_OK;
}

void mxattn_set_debug_flags(uint32_t flags) { g_debug_flags = flags; }

const char* mxattn_last_error(void) { return t_err; }

}  // extern "C"
