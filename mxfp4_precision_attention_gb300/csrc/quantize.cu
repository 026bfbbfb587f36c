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

#include <cmath>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace mxattn {
namespace {

constexpr float kRotScale = 0x1.6a09e6p-4f;  // binary32 nearest to 2^-3.5 = 1/sqrt(128)

// Block scale exponent for a finite block maximum M > 0, M = 1.f * 2^(b-127):
//   UOS  ceil(log2(M/7.25)) = (b-126) - 3 if 1.f <= 1.8125 else (b-126) - 2
//   TFS  ceil(log2(M/6))    = (b-126) - 3 if 1.f <= 1.5    else (b-126) - 2
//   OCP  floor(log2 M) - 2  = (b-126) - 3
//   ceil(log2(M/q)), q in (4, 8]: (b-126) - 3 if 1.f <= q/4 else (b-126) - 2,
//        and one lower for an exact power of two when q = 8
// i.e. one comparison of the mantissa field against mant_thr (0x680000,
// 0x400000, floor((q/4 - 1) * 2^23), or 0x7FFFFF so that it always holds).
// Denormal maxima and anything below the E8M0 range clamp to -127.
struct ScaleRule {
  uint32_t mant_thr;
  uint32_t pow2_down;  // q = 8: M = 2^k gives e = k - 3
};

__device__ __forceinline__ int block_exponent(float M, ScaleRule r) {
  const uint32_t bits = __float_as_uint(M);
  const int b = static_cast<int>(bits >> 23);
  if (b == 0) return -127;
  const uint32_t mant = bits & 0x7FFFFFu;
  const int e = b - 126 - (mant <= r.mant_thr ? 3 : 2) - ((r.pow2_down && mant == 0u) ? 1 : 0);
  return e < -127 ? -127 : e;
}

ScaleRule make_rule(int rule, double qmax) {
  ScaleRule r{0x680000u, 0u};
  if (rule == kRuleOCP) r.mant_thr = 0x7FFFFFu;
  if (rule == kRuleTFS) r.mant_thr = 0x400000u;
  if (rule == kRuleCeilQ) {
    const double t = std::floor((qmax / 4.0 - 1.0) * 8388608.0);  // exact: qmax/4 - 1 has qmax's ulp
    r.mant_thr = t >= 8388607.0 ? 0x7FFFFFu : static_cast<uint32_t>(t);
    r.pow2_down = qmax >= 8.0 ? 1u : 0u;
  }
  return r;
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
// Four lanes per token. Lane l holds the 8-channel chunks c = 4k + l
// (k = 0..3), i.e. z[8k + i] is channel 8(4k + l) + i. In this layout the
// butterflies h = 1, 2, 4 (inside a chunk) and h = 32, 64 (chunk k ^ 1,
// k ^ 2) stay in the lane; only h = 8 and h = 16 pair lanes l ^ 1 and l ^ 2.
// Each load instruction reads whole 64-byte segments of 8 token rows.
constexpr int kQkThreads = 256;
constexpr int kQkLanesPerToken = 4;

// One butterfly on a register pair: (a, b) -> (a + b, a - b) in binary32.
__device__ __forceinline__ void bfly(float& a, float& b) {
  const float s = __fadd_rn(a, b), d = __fsub_rn(a, b);
  a = s;
  b = d;
}
// Two butterflies at once: (a0,a1), (b0,b1) -> (a + b, a - b) per component.
// a - b is formed as fma(b, -1, a): the product is exact, so it rounds once,
// exactly like a subtraction.
__device__ __forceinline__ void bfly2(float& a0, float& a1, float& b0, float& b1) {
  const float2 a = make_float2(a0, a1), b = make_float2(b0, b1);
  const float2 s = __fadd2_rn(a, b), d = __ffma2_rn(b, make_float2(-1.0f, -1.0f), a);
  a0 = s.x;
  a1 = s.y;
  b0 = d.x;
  b1 = d.y;
}

__global__ void __launch_bounds__(kQkThreads) rotate_quantize_qk_kernel(const uint4* __restrict__ x,
                                                                         uint32_t* __restrict__ codes,
                                                                         uint32_t* __restrict__ scales,
                                                                         int64_t BH, int64_t N, int64_t NT,
                                                                         ScaleRule rule, int rotate) {
  const int lane = threadIdx.x & 31;
  const int l = lane & 3;
  const int64_t slots_per_head = NT * kTile;
  const int64_t total_slots = BH * slots_per_head;
  constexpr int kTokPerWarp = 32 / kQkLanesPerToken;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (kQkThreads / 32);
  // h = 8, 16: the lane holding the lower channel of the pair adds, the other subtracts
  const float sgn8 = (l & 1) ? -1.0f : 1.0f, sgn16 = (l & 2) ? -1.0f : 1.0f;
  for (int64_t grp = static_cast<int64_t>(blockIdx.x) * (kQkThreads / 32) + threadIdx.x / 32;
       grp * kTokPerWarp < total_slots; grp += warps_total) {
    const int64_t slot = grp * kTokPerWarp + lane / kQkLanesPerToken;
    const bool in_range = slot < total_slots;
    const int64_t bh = in_range ? slot / slots_per_head : 0;
    const int64_t n = in_range ? slot - bh * slots_per_head : 0;
    const bool real = in_range && n < N;
    float z[32];
    if (real) {
      const uint4* row = x + (bh * N + n) * 16;
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const uint4 raw = ld_nc_v4(row + 4 * k + l);
        bf16x2_to_f32(raw.x, z[8 * k + 0], z[8 * k + 1]);
        bf16x2_to_f32(raw.y, z[8 * k + 2], z[8 * k + 3]);
        bf16x2_to_f32(raw.z, z[8 * k + 4], z[8 * k + 5]);
        bf16x2_to_f32(raw.w, z[8 * k + 6], z[8 * k + 7]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; i++) z[i] = 0.0f;
    }
    if (rotate) {
#pragma unroll
      for (int k = 0; k < 4; k++) {
        float* c = z + 8 * k;
        // h = 1
        bfly(c[0], c[1]);
        bfly(c[2], c[3]);
        bfly(c[4], c[5]);
        bfly(c[6], c[7]);
        // h = 2
        bfly2(c[0], c[1], c[2], c[3]);
        bfly2(c[4], c[5], c[6], c[7]);
        // h = 4
        bfly2(c[0], c[1], c[4], c[5]);
        bfly2(c[2], c[3], c[6], c[7]);
      }
      // h = 8 (lane ^ 1), h = 16 (lane ^ 2): new = own * sign + partner
#pragma unroll
      for (int st = 0; st < 2; st++) {
        const int mask = st ? 2 : 1;
        const float sg = st ? sgn16 : sgn8;
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float p0 = __shfl_xor_sync(0xffffffffu, z[i], mask);
          const float p1 = __shfl_xor_sync(0xffffffffu, z[i + 1], mask);
          const float2 r = __ffma2_rn(make_float2(z[i], z[i + 1]), make_float2(sg, sg), make_float2(p0, p1));
          z[i] = r.x;
          z[i + 1] = r.y;
        }
      }
      // h = 32 (chunk k ^ 1), h = 64 (chunk k ^ 2)
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        bfly2(z[i], z[i + 1], z[8 + i], z[9 + i]);
        bfly2(z[16 + i], z[17 + i], z[24 + i], z[25 + i]);
      }
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        bfly2(z[i], z[i + 1], z[16 + i], z[17 + i]);
        bfly2(z[8 + i], z[9 + i], z[24 + i], z[25 + i]);
      }
      const float2 rs = make_float2(kRotScale, kRotScale);
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float2 r = __fmul2_rn(make_float2(z[i], z[i + 1]), rs);
        z[i] = r.x;
        z[i + 1] = r.y;
      }
    }
    // block k = channels 32k .. 32k+31 = chunk k of the token's four lanes
    uint32_t sw = 0;
#pragma unroll
    for (int k = 0; k < 4; k++) {
      const float* c = z + 8 * k;
      float m = fmaxf(fmaxf(fmaxf(fabsf(c[0]), fabsf(c[1])), fmaxf(fabsf(c[2]), fabsf(c[3]))),
                      fmaxf(fmaxf(fabsf(c[4]), fabsf(c[5])), fmaxf(fabsf(c[6]), fabsf(c[7]))));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      uint32_t word = 0;
      uint32_t sbyte = 127;
      if (m > 0.0f) {
        const int e = block_exponent(m, rule);
        const float2 inv = make_float2(pow2_neg(e), pow2_neg(e));
        const float2 a = __fmul2_rn(make_float2(c[0], c[1]), inv), b = __fmul2_rn(make_float2(c[2], c[3]), inv);
        const float2 cc = __fmul2_rn(make_float2(c[4], c[5]), inv), d = __fmul2_rn(make_float2(c[6], c[7]), inv);
        word = pack_e2m1x8(a.x, a.y, b.x, b.y, cc.x, cc.y, d.x, d.y);
        sbyte = static_cast<uint32_t>(e + 127);
      }
      if (real) codes[(bh * N + n) * 16 + 4 * k + l] = word;
      sw |= sbyte << (8 * k);
    }
    if (in_range && l == 0) {
      const int64_t t = n / kTile;
      const int r = static_cast<int>(n - t * kTile);
      scales[(bh * NT + t) * (kSfAtomBytes / 4) + (r % 32) * 4 + (r / 32)] = sw;
    }
  }
}

// ----------------------------------------------------------------- (b)
// One CTA per (head, 128-token tile), eight warps. Warp w takes token block
// w/2 (32 tokens) of channel half w%2 (64 channels); lane l owns channels
// c0 = 64*(w%2) + 2l and c0 + 1, i.e. the l-th bf16x2 word of the half row.
// Each load instruction reads 128 contiguous bytes of one token row; a lane
// ends up with its two channels' whole 32-token block, so block maxima and
// codes need no exchange between threads. Only the scale atom is assembled in
// shared memory.
constexpr int kVThreads = 256;

__global__ void __launch_bounds__(kVThreads, 3) quantize_v_kernel(const uint32_t* __restrict__ v,
                                                                   uint8_t* __restrict__ codes,
                                                                   uint32_t* __restrict__ scales, int64_t N,
                                                                   int64_t NT, int64_t row_bytes, ScaleRule rule) {
  __shared__ uint32_t atom[kSfAtomBytes / 4];
  const int64_t t = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int half = warp & 1, kb = warp >> 1;
  const int c0 = 64 * half + 2 * lane;
  const int64_t tok0 = t * kTile + kb * kBlock;
  const uint32_t* src = v + (bh * N + tok0) * (kD / 2) + 32 * half + lane;
  uint32_t w[kBlock];
#pragma unroll
  for (int i = 0; i < kBlock; i++) w[i] = tok0 + i < N ? __ldg(src + i * (kD / 2)) : 0u;
  // |.| maxima of both channels at once: bf16 max is exact
  uint32_t mw = w[0] & 0x7FFF7FFFu;
#pragma unroll
  for (int i = 1; i < kBlock; i++) {
    const uint32_t a = w[i] & 0x7FFF7FFFu;
    asm("max.bf16x2 %0, %0, %1;" : "+r"(mw) : "r"(a));
  }
  float lo_m, hi_m;
  bf16x2_to_f32(mw, lo_m, hi_m);
  const float m2[2] = {lo_m, hi_m};
  uint32_t sb[2];
  float inv[2];
#pragma unroll
  for (int h = 0; h < 2; h++) {
    const bool nz = m2[h] > 0.0f;
    const int e = nz ? block_exponent(m2[h], rule) : 0;
    sb[h] = nz ? static_cast<uint32_t>(e + 127) : 127u;
    inv[h] = nz ? pow2_neg(e) : 0.0f;
  }
  uint32_t cw[2][4];
  const float2 inv2 = make_float2(inv[0], inv[1]);
#pragma unroll
  for (int g = 0; g < 4; g++) {
    float q0[8], q1[8];
#pragma unroll
    for (int i = 0; i < 8; i++) {
      float lo, hi;
      bf16x2_to_f32(w[8 * g + i], lo, hi);
      const float2 q = __fmul2_rn(make_float2(lo, hi), inv2);
      q0[i] = q.x;
      q1[i] = q.y;
    }
    cw[0][g] = pack_e2m1x8(q0[0], q0[1], q0[2], q0[3], q0[4], q0[5], q0[6], q0[7]);
    cw[1][g] = pack_e2m1x8(q1[0], q1[1], q1[2], q1[3], q1[4], q1[5], q1[6], q1[7]);
  }
  if (tok0 < N) {  // block holds at least one real token; it lies inside Npad
#pragma unroll
    for (int h = 0; h < 2; h++)
      *reinterpret_cast<uint4*>(codes + (bh * kD + c0 + h) * row_bytes + tok0 / 2) =
          make_uint4(cw[h][0], cw[h][1], cw[h][2], cw[h][3]);
  }
  // scale byte of row c, block kb -> (c%32)*16 + (c/32)*4 + kb
  uint8_t* ab = reinterpret_cast<uint8_t*>(atom);
#pragma unroll
  for (int h = 0; h < 2; h++) {
    const int c = c0 + h;
    ab[(c % 32) * 16 + (c / 32) * 4 + kb] = static_cast<uint8_t>(sb[h]);
  }
  __syncthreads();
  if (threadIdx.x < kSfAtomBytes / 16)
    reinterpret_cast<uint4*>(scales + (bh * NT + t) * (kSfAtomBytes / 4))[threadIdx.x] =
        reinterpret_cast<const uint4*>(atom)[threadIdx.x];
}

}  // namespace

void rule_threshold(int rule, double qmax, uint32_t* mant_thr, uint32_t* pow2_down) {
  const ScaleRule r = make_rule(rule, qmax);
  *mant_thr = r.mant_thr;
  *pow2_down = r.pow2_down;
}

cudaError_t launch_rotate_quantize_qk(const void* x, int64_t BH, int64_t N, void* codes, void* scales, int rule,
                                      double qmax, int rotate, cudaStream_t s) {
  const int64_t NT = ceil_div(N, kTile);
  const int64_t groups = ceil_div(BH * NT * kTile, 32 / kQkLanesPerToken);  // one warp-iteration each
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = ceil_div(groups, kQkThreads / 32);
  const int grid = static_cast<int>(want < sms * 8 ? want : sms * 8);
  rotate_quantize_qk_kernel<<<grid, kQkThreads, 0, s>>>(static_cast<const uint4*>(x),
                                                        static_cast<uint32_t*>(codes),
                                                        static_cast<uint32_t*>(scales), BH, N, NT,
                                                        make_rule(rule, qmax), rotate);
  return cudaGetLastError();
}

cudaError_t launch_quantize_v(const void* v, int64_t BH, int64_t N, void* codes, void* scales, int rule,
                              double qmax, cudaStream_t s) {
  const int64_t NT = ceil_div(N, kTile);
  const int64_t row_bytes = ceil_div(N, kBlock) * kBlock / 2;
  dim3 grid(static_cast<unsigned>(NT), static_cast<unsigned>(BH));
  quantize_v_kernel<<<grid, kVThreads, 0, s>>>(static_cast<const uint32_t*>(v), static_cast<uint8_t*>(codes),
                                               static_cast<uint32_t*>(scales), N, NT, row_bytes,
                                               make_rule(rule, qmax));
  return cudaGetLastError();
}

}  // namespace mxattn
