// MXFP4 quantizers of the MXAttention forward ("MXAttention", the rotation
// and quantization steps of Algorithm 2 in section 4.3, with the UOS block
// quantizer of Algorithm 1).
//
//  (a) rotate_quantize_qk: per token, Hadamard-rotate the 128 channels
//      (binary32 butterflies h = 1,2,...,64, then x 2^-3.5 rounded to binary32)
//      and quantize each 32-channel block to E2M1 with the UOS scale
//      e = ceil(log2(M / 7.25)). The ablation variants (section 5.4, Table 3)
//      skip the rotation and/or use the OCP scale e = floor(log2 M) - 2
//      (Eq. 11) or the TFS scale e = ceil(log2(M / 6)) (Eq. 14).
//  (b) quantize_v: per channel, quantize blocks of 32 consecutive tokens
//      (blocks counted from token 0, last block zero-padded) and store the codes
//      transposed (token-contiguous), the K-major layout the P.V MMA reads.
//
// Output layouts (bytes):
//   Q/K codes   [BH][N][64]               element 2j in the low nibble of byte j
//   V codes     [BH][128][Npad/2]         Npad = 32*ceil(N/32); token 2j low nibble
//   scales      [BH][ceil(N/128)][512]    one 512-byte atom per 128-row tile:
//               row r of the tile, block k -> byte (r%32)*16 + (r/32)*4 + k
//               (rows = tokens for Q/K, channels for V; blocks = channel blocks
//               for Q/K, token blocks for V). Rows or blocks past N hold 127.
//   scale byte = e + 127 (E8M0); an all-zero block gets 127 and zero codes.
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace mxattn {
namespace {

constexpr float kRotScale = 0x1.6a09e6p-4f;  // binary32 nearest to 2^-3.5 = 1/sqrt(128)

// Block scale exponent for a finite block maximum M > 0, M = 1.f * 2^(b-127):
//   UOS  ceil(log2(M/7.25)) = (b-126) - 3 if 1.f <= 1.8125 else (b-126) - 2
//   TFS  ceil(log2(M/6))    = (b-126) - 3 if 1.f <= 1.5    else (b-126) - 2
//   OCP  floor(log2 M) - 2  = (b-126) - 3
// i.e. one comparison of the mantissa field against mant_thr (0x680000,
// 0x400000, or 0x7FFFFF so that it always holds). Denormal maxima and
// anything below the E8M0 range clamp to -127.
__device__ __forceinline__ int block_exponent(float M, uint32_t mant_thr) {
  const uint32_t bits = __float_as_uint(M);
  const int b = static_cast<int>(bits >> 23);
  if (b == 0) return -127;
  const int e = b - 126 - ((bits & 0x7FFFFFu) <= mant_thr ? 3 : 2);
  return e < -127 ? -127 : e;
}

uint32_t rule_mantissa_threshold(int rule) {
  return rule == kRuleOCP ? 0x7FFFFFu : (rule == kRuleTFS ? 0x400000u : 0x680000u);
}

// 2^-e as binary32; valid for e in [-127, 126], which covers every finite M.
__device__ __forceinline__ float pow2_neg(int e) { return __uint_as_float(static_cast<uint32_t>(127 - e) << 23); }

__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xFFFF0000u);
}

__device__ __forceinline__ uint4 ld_nc_v4(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// ----------------------------------------------------------------- (a)
// 16 lanes per token, 8 consecutive channels per lane (channel 8*l + i).
// Butterflies h = 1, 2, 4 are in-lane; h = 8..64 pair lanes l and l^(h/8).
constexpr int kQkThreads = 256;

__global__ void __launch_bounds__(kQkThreads) rotate_quantize_qk_kernel(const uint4* __restrict__ x,
                                                                         uint32_t* __restrict__ codes,
                                                                         uint32_t* __restrict__ scales,
                                                                         int64_t BH, int64_t N, int64_t NT,
                                                                         uint32_t mant_thr, int rotate) {
  const int lane = threadIdx.x & 31;
  const int l = lane & 15;
  const int64_t slots_per_head = NT * kTile;
  const int64_t total_slots = BH * slots_per_head;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (kQkThreads / 32);
  for (int64_t pair = static_cast<int64_t>(blockIdx.x) * (kQkThreads / 32) + threadIdx.x / 32;
       pair * 2 < total_slots; pair += warps_total) {
    const int64_t slot = pair * 2 + (lane >> 4);
    const bool in_range = slot < total_slots;
    const int64_t bh = in_range ? slot / slots_per_head : 0;
    const int64_t n = in_range ? slot - bh * slots_per_head : 0;
    const bool real = in_range && n < N;
    float z[8];
    if (real) {
      const uint4 raw = ld_nc_v4(x + (bh * N + n) * 16 + l);
      bf16x2_to_f32(raw.x, z[0], z[1]);
      bf16x2_to_f32(raw.y, z[2], z[3]);
      bf16x2_to_f32(raw.z, z[4], z[5]);
      bf16x2_to_f32(raw.w, z[6], z[7]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; i++) z[i] = 0.0f;
    }
    if (rotate) {
    // in-lane butterflies: h = 1, 2, 4
#pragma unroll
    for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
      for (int i = 0; i < 8; i++) {
        if (i & h) continue;
        const float a = z[i], b = z[i + h];
        z[i] = __fadd_rn(a, b);
        z[i + h] = __fsub_rn(a, b);
      }
    }
    // cross-lane butterflies: h = 8, 16, 32, 64 <-> lane xor 1, 2, 4, 8
#pragma unroll
    for (int s = 1; s < 16; s <<= 1) {
      const bool upper = (l & s) != 0;
#pragma unroll
      for (int i = 0; i < 8; i++) {
        const float p = __shfl_xor_sync(0xffffffffu, z[i], s);
        z[i] = upper ? __fsub_rn(p, z[i]) : __fadd_rn(z[i], p);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; i++) z[i] = __fmul_rn(z[i], kRotScale);
    }
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++) m = fmaxf(m, fabsf(z[i]));
    // block = 32 channels = lanes 4b..4b+3 of the token
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    uint32_t word = 0;
    uint32_t sbyte = 127;
    if (m > 0.0f) {
      const int e = block_exponent(m, mant_thr);
      const float inv = pow2_neg(e);
      word = pack_e2m1x8(__fmul_rn(z[0], inv), __fmul_rn(z[1], inv), __fmul_rn(z[2], inv),
                         __fmul_rn(z[3], inv), __fmul_rn(z[4], inv), __fmul_rn(z[5], inv),
                         __fmul_rn(z[6], inv), __fmul_rn(z[7], inv));
      sbyte = static_cast<uint32_t>(e + 127);
    }
    if (real) codes[(bh * N + n) * 16 + l] = word;
    uint32_t sw = sbyte << (8 * (l >> 2));
    sw |= __shfl_xor_sync(0xffffffffu, sw, 4);
    sw |= __shfl_xor_sync(0xffffffffu, sw, 8);
    if (in_range && l == 0) {
      const int64_t t = n / kTile;
      const int r = static_cast<int>(n - t * kTile);
      scales[(bh * NT + t) * (kSfAtomBytes / 4) + (r % 32) * 4 + (r / 32)] = sw;
    }
  }
}

// ----------------------------------------------------------------- (b)
// One CTA per (head, 128-token tile); thread c owns channel c.
constexpr int kVThreads = 128;
constexpr int kVRowWords = kD / 2 + 1;  // bf16x2 words per staged token row (+1 pad)

__global__ void __launch_bounds__(kVThreads) quantize_v_kernel(const uint4* __restrict__ v,
                                                                uint8_t* __restrict__ codes,
                                                                uint32_t* __restrict__ scales, int64_t N,
                                                                int64_t NT, int64_t row_bytes, uint32_t mant_thr) {
  __shared__ uint32_t tile[kTile * kVRowWords];
  const int64_t t = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int tid = threadIdx.x;
  const int64_t n0 = t * kTile;
  // stage 128 tokens x 128 channels (16-byte coalesced loads; tokens >= N read as 0)
#pragma unroll 4
  for (int i = tid; i < kTile * 16; i += kVThreads) {
    const int row = i / 16, q = i % 16;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (n0 + row < N) val = ld_nc_v4(v + (bh * N + n0 + row) * 16 + q);
    uint32_t* dst = tile + row * kVRowWords + q * 4;
    dst[0] = val.x;
    dst[1] = val.y;
    dst[2] = val.z;
    dst[3] = val.w;
  }
  __syncthreads();
  const int c = tid;
  const int word = c >> 1;
  const bool hi_half = (c & 1) != 0;
  uint32_t sw = 0;
#pragma unroll
  for (int kb = 0; kb < kTile / kBlock; kb++) {
    float val[kBlock];
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < kBlock; i++) {
      const uint32_t w = tile[(kb * kBlock + i) * kVRowWords + word];
      val[i] = hi_half ? __uint_as_float(w & 0xFFFF0000u) : __uint_as_float(w << 16);
      m = fmaxf(m, fabsf(val[i]));
    }
    uint32_t sbyte = 127;
    uint4 packed = make_uint4(0, 0, 0, 0);
    if (m > 0.0f) {
      const int e = block_exponent(m, mant_thr);
      const float inv = pow2_neg(e);
      uint32_t w4[4];
#pragma unroll
      for (int g = 0; g < 4; g++) {
        w4[g] = pack_e2m1x8(__fmul_rn(val[8 * g + 0], inv), __fmul_rn(val[8 * g + 1], inv),
                            __fmul_rn(val[8 * g + 2], inv), __fmul_rn(val[8 * g + 3], inv),
                            __fmul_rn(val[8 * g + 4], inv), __fmul_rn(val[8 * g + 5], inv),
                            __fmul_rn(val[8 * g + 6], inv), __fmul_rn(val[8 * g + 7], inv));
      }
      packed = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      sbyte = static_cast<uint32_t>(e + 127);
    }
    sw |= sbyte << (8 * kb);
    const int64_t tok0 = n0 + kb * kBlock;
    if (tok0 < N) {  // block holds at least one real token; it lies inside Npad
      *reinterpret_cast<uint4*>(codes + (bh * kD + c) * row_bytes + tok0 / 2) = packed;
    }
  }
  scales[(bh * NT + t) * (kSfAtomBytes / 4) + (c % 32) * 4 + (c / 32)] = sw;
}

}  // namespace

cudaError_t launch_rotate_quantize_qk(const void* x, int64_t BH, int64_t N, void* codes, void* scales, int rule,
                                      int rotate, cudaStream_t s) {
  const int64_t NT = ceil_div(N, kTile);
  const int64_t pairs = ceil_div(BH * NT * kTile, 2);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = ceil_div(pairs, kQkThreads / 32);
  const int grid = static_cast<int>(want < sms * 8 ? want : sms * 8);
  rotate_quantize_qk_kernel<<<grid, kQkThreads, 0, s>>>(static_cast<const uint4*>(x),
                                                        static_cast<uint32_t*>(codes),
                                                        static_cast<uint32_t*>(scales), BH, N, NT,
                                                        rule_mantissa_threshold(rule), rotate);
  return cudaGetLastError();
}

cudaError_t launch_quantize_v(const void* v, int64_t BH, int64_t N, void* codes, void* scales, int rule,
                              cudaStream_t s) {
  const int64_t NT = ceil_div(N, kTile);
  const int64_t row_bytes = ceil_div(N, kBlock) * kBlock / 2;
  dim3 grid(static_cast<unsigned>(NT), static_cast<unsigned>(BH));
  quantize_v_kernel<<<grid, kVThreads, 0, s>>>(static_cast<const uint4*>(v), static_cast<uint8_t*>(codes),
                                               static_cast<uint32_t*>(scales), N, NT, row_bytes,
                                               rule_mantissa_threshold(rule));
  return cudaGetLastError();
}

}  // namespace mxattn
