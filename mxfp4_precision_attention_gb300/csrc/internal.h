// Host-side declarations shared by the CUDA translation units of libmxattn.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mxattn {

constexpr int kD = 128;        // head dimension supported by every kernel
constexpr int kBlock = 32;     // MX block size (elements sharing one E8M0 scale)
constexpr int kTile = 128;     // query rows / key columns per tile (Bc)
constexpr int kSfAtomBytes = 512;  // scale bytes per 128-row tile (128 rows x 4 blocks)

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Debug switches read by the attention kernels (set through the C ABI).
enum : uint32_t { kDebugNeverArriveS = 1u };

// Block scale rules (same numbering as mxattn_scale_rule) and l placements.
enum : int { kRuleUOS = 0, kRuleOCP = 1, kRuleTFS = 2, kRuleCeilQ = 3 };
enum : int { kPlacePNQ = 0, kPlaceDirect = 1 };

// Mantissa-field threshold of a block scale rule (see quantize.cu): the
// exponent of a block maximum M = 1.f * 2^(b-127) is (b-126) - 3 if the
// mantissa field is <= mant_thr, else (b-126) - 2, and one lower for an exact
// power of two when pow2_down is set.
void rule_threshold(int rule, double qmax, uint32_t* mant_thr, uint32_t* pow2_down);

// One tensor of a quantizer launch: bf16 [BH][N][128] in, codes and scales
// out (layouts in quantize.cu). qmax is used by kRuleCeilQ only (a value in
// (4, 8]); rotate applies to Q/K jobs only.
struct QuantizeJob {
  const void* x;
  void* codes;
  void* scales;
  int rule;
  double qmax;
  int is_v;
  int rotate;
  float* amax;  // non-null: NVFP4 (16-element blocks, E4M3 scales), tensor max |x| written here
};
// Up to three jobs of the same B*H and N in one launch (their tiles interleave).
cudaError_t launch_quantize(const QuantizeJob* jobs, int njobs, int64_t BH, int64_t N, cudaStream_t s);
cudaError_t launch_rotate_quantize_qk(const void* x, int64_t BH, int64_t N, void* codes, void* scales, int rule,
                                      double qmax, int rotate, cudaStream_t s);
cudaError_t launch_quantize_v(const void* v, int64_t BH, int64_t N, void* codes, void* scales, int rule,
                              double qmax, cudaStream_t s);

struct Mxfp4FwdArgs {
  const void* q_codes;
  const void* q_scales;
  const void* k_codes;
  const void* k_scales;
  const void* v_codes;
  const void* v_scales;
  const void* v_bf16;  // causal diagonal blocks
  int64_t BH, N;
  int causal;  // 0, 1, or 2: diagonal V block re-quantized over the prefix (variant kernel)
  float* out;
  void* out_bf16;        // non-null (and out null): O / l written as bf16 [BH][N][128] here
  uint8_t* phat_codes;   // optional diagnostic dump, [BH][N][ceil(N/128)*64]
  uint8_t* phat_scales;  // optional diagnostic dump, [BH][N][ceil(N/128)*4]
  uint32_t debug_flags;
  int p_rule;     // scale rule of the P~ blocks (kRule*)
  double p_qmax;  // Q_max of kRuleCeilQ
  int placement;  // kPlacePNQ: l from P^ (Eq. 47); kPlaceDirect: l from P~ (Eq. 16)
  // NVFP4 operands (all three non-null, or all null for MXFP4): the tensors'
  // max |x| from the NVFP4 quantizers; scales are then two E4M3 atoms per tile
  const float* q_amax;
  const float* k_amax;
  const float* v_amax;
};
cudaError_t launch_mxfp4_forward(const Mxfp4FwdArgs& a, cudaStream_t s);

struct Bf16FwdArgs {
  const void* q;  // bf16 [BH][Nq][128]
  const void* k;  // bf16 [BH][Nk][128]
  const void* v;  // bf16 [BH][Nk][128]
  int64_t BH, Nq, Nk;
  int causal;
  float* out;
  uint32_t debug_flags;
};
cudaError_t launch_bf16_forward(const Bf16FwdArgs& a, cudaStream_t s);

// Tensor-core rate probe (mma_rate.cu): one CTA per SM, `iters` pairs of
// M128 Nn K64 kind::mxf4 MMAs each (n = 128 or 256); *ctas_out = the grid size.
cudaError_t launch_mxf4_mma_rate(int64_t iters, int n, float* d_out, int* ctas_out, cudaStream_t s);
double mxf4_mma_rate_flops(int64_t iters, int n, int ctas);

// Device status word written by kernels whose bounded waits expired.
cudaError_t read_and_clear_device_status(int* status, cudaStream_t s);
int* device_status_ptr();

// Replace the calling thread's mxattn_last_error() message.
void set_last_error(const char* msg);

// cuTensorMapEncodeTiled through the runtime's driver entry point.
bool encode_tensor_map(void* map, int dtype_is_bf16, int rank, void* base, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box, int swizzle_bytes);

}  // namespace mxattn
