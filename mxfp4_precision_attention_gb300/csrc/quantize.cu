// MXFP4 quantizers of the MXAttention forward ("MXAttention", the rotation
// and quantization steps of Algorithm 2 in section 4.3, with the UOS block
// quantizer of Algorithm 1).
//
// One launch per call. The single-tensor calls, the ablation rules and NVFP4
// run quantize_tiles_kernel; mxattn_quantize_qkv (the forward's Q, K and V,
// MXFP4) runs quantize_qkv_roles_kernel, the same per-tile code with the
// work split by role among three warpgroups.
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
#include <cuda.h>
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

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// max |v[i]| over 32 values
__device__ __forceinline__ float absmax32(const float* v) {
  float a[11];
#pragma unroll
  for (int i = 0; i < 10; i++) a[i] = max3f(fabsf(v[3 * i]), fabsf(v[3 * i + 1]), fabsf(v[3 * i + 2]));
  a[10] = fmaxf(fabsf(v[30]), fabsf(v[31]));
  const float b0 = max3f(a[0], a[1], a[2]), b1 = max3f(a[3], a[4], a[5]), b2 = max3f(a[6], a[7], a[8]);
  return max3f(max3f(b0, b1, b2), a[9], a[10]);
}

__device__ __forceinline__ void record_error(int* status, int code, volatile int* abort_flag) {
  *abort_flag = 1;
  atomicCAS(status, 0, code);
}

// ----------------------------------------------------------------- kernel
// One persistent kernel serves every quantizer call. A work unit is one
// 128-token tile of one head of one tensor: 128 rows of 256 bytes, brought
// into shared memory by two TMA loads (channels 0-63 and 64-127; 128 bytes
// per row each, 128-byte swizzle: 16-byte chunk c of row r sits at chunk
// c ^ (r % 8)), into a ring of kQStages buffers. All four warps quantize;
// thread 0 also refills the ring: once every warp has read unit i-1 into
// registers, it loads unit i-1+kQStages into that buffer. Units of up to
// three tensors (Q, K, V of one call) interleave, so the rotation's ALU work
// and the V tiles' light work share the SMs.
//
//  (a) Q/K tile: one thread per token, its 128 channels in registers in
//      natural order. The h = 1 butterflies pair the halves of a register
//      pair (scalar adds); h = 2 ... 64 pair register pair (i, i+1) with
//      (i+h, i+h+1) (packed f32x2 adds). Same binary32 operations in the same
//      stage order as the plain definition.
//  (b) V tile: warp w takes token block w (32 tokens); lane l owns channels
//      2l, 2l+1, 64+2l, 65+2l (word l of each half row), so every block
//      maximum and code is formed inside the thread.
// Two CTAs of four warps per SM: a Q/K thread holds a token's 128 channels
// (192 registers, no spills), and the register file is split per SMSP
// (16K each), so two 4-warp CTAs (two warps per SMSP) is the most that fits;
// three 32 KB stages each keep six tiles in flight per SM.
constexpr int kQStages = 3;
constexpr int kQMinBlocks = 2;
constexpr int kQThreads = 128;  // four warps; thread 0 also issues the loads
constexpr int kQConsumers = 128;
constexpr uint32_t kQHalfBytes = kTile * 128;        // one TMA box: 128 rows x 64 channels
constexpr uint32_t kQStageBytes = 2 * kQHalfBytes;   // 32 KB
constexpr uint32_t kQSmemBytes = kQStages * kQStageBytes + 2 * kQStages * 8 + 16 + 1024;

struct QTensor {
  uint8_t* codes;
  uint32_t* scales;
  ScaleRule rule;
  int is_v;    // 0: Q/K (per-token channel blocks), 1: V (per-channel token blocks)
  int rotate;  // Q/K only
  int nv;      // 1: NVFP4 (16-element blocks, E4M3 scales; no rotation)
  const float* amax;  // NVFP4: the tensor's max |x| (written by the amax pass)
};
struct QParams {
  QTensor t[3];
  int ntensors;
  int64_t BH, N, NT, row_bytes;  // row_bytes: V codes per channel row (Npad/2)
  int64_t units;                 // ntensors * BH * NT
  int* status;
};

// ----------------------------------------------------------------- NVFP4
// NVFP4 ("MXAttention" section 1: E2M1 values in 16-element blocks, an E4M3
// block scale and a tensor-level scale) with the binary32 order of operations
// the comparison baseline fixes:
//   e_t = fl(2688 / amax)  (2688 = 6 * 448; 1 for an all-zero tensor)
//   sc  = E4M3(fl(fl(M / 6) * e_t)), round to nearest even, saturating at 448
//   sc == 0: every code 0; else k = fl(e_t / value(sc)), code = E2M1(fl(x * k))
// Scales: two 512-byte atoms per 128-row tile, atom kk holding blocks
// 4kk .. 4kk+3 (the K range of one 64-wide MMA) at byte
// (r%32)*16 + (r/32)*4 + (block % 4).
__device__ __forceinline__ float nv_encode(const float* amax) {
  const float a = __ldg(amax);
  return a > 0.0f ? __fdiv_rn(2688.0f, a) : 1.0f;
}

// E4M3 code (round to nearest even, saturating at 448) of v >= 0.
__device__ __forceinline__ uint32_t e4m3_code(float v) {
  uint16_t h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(0.0f), "f"(v));
  return h & 0xFFu;
}

// Value of a finite nonnegative E4M3 code.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t ef = (c >> 3) & 15u, m = c & 7u;
  return ef ? __uint_as_float(((ef + 120u) << 23) | (m << 20)) : static_cast<float>(m) * 0x1p-9f;
}

// Block scale code and element factor of a block maximum M.
__device__ __forceinline__ uint32_t nv_block_scale(float M, float et, float* k) {
  const uint32_t sc = e4m3_code(__fmul_rn(__fdiv_rn(M, 6.0f), et));
  *k = sc ? __fdiv_rn(et, e4m3_value(sc)) : 0.0f;
  return sc;
}

__device__ __forceinline__ float absmax16(const float* v) {
  const float a0 = max3f(fabsf(v[0]), fabsf(v[1]), fabsf(v[2])), a1 = max3f(fabsf(v[3]), fabsf(v[4]), fabsf(v[5]));
  const float a2 = max3f(fabsf(v[6]), fabsf(v[7]), fabsf(v[8])), a3 = max3f(fabsf(v[9]), fabsf(v[10]), fabsf(v[11]));
  const float a4 = max3f(fabsf(v[12]), fabsf(v[13]), fabsf(v[14]));
  return max3f(max3f(a0, a1, a2), max3f(a3, a4, fabsf(v[15])), 0.0f);
}

// NVFP4 Q/K tile: one thread per token, 8 blocks of 16 channels.
__device__ __forceinline__ void quantize_qk_tile_nv(const uint8_t* tile, int r, int64_t bh, int64_t t,
                                                    const QParams& p, const QTensor& T, uint32_t empty_bar) {
  float z[kD];
#pragma unroll
  for (int c = 0; c < kD / 8; c++) {
    const uint4 raw = *reinterpret_cast<const uint4*>(tile + (c >> 3) * kQHalfBytes + r * 128 +
                                                      (((c & 7) ^ (r & 7)) << 4));
    bf16x2_to_f32(raw.x, z[8 * c + 0], z[8 * c + 1]);
    bf16x2_to_f32(raw.y, z[8 * c + 2], z[8 * c + 3]);
    bf16x2_to_f32(raw.z, z[8 * c + 4], z[8 * c + 5]);
    bf16x2_to_f32(raw.w, z[8 * c + 6], z[8 * c + 7]);
  }
  __syncwarp();
  if ((r & 31) == 0) mbar_arrive(empty_bar);
  const float et = nv_encode(T.amax);
  const int64_t n = t * kTile + r;
  const bool real = n < p.N;
  uint2* crow = reinterpret_cast<uint2*>(T.codes) + (bh * p.N + n) * (kD / 16);
  uint32_t sw[2] = {0u, 0u};
#pragma unroll
  for (int b = 0; b < kD / 16; b++) {
    const float* c = z + 16 * b;
    float k;
    const uint32_t sc = nv_block_scale(absmax16(c), et, &k);
    uint32_t w[2];
#pragma unroll
    for (int g = 0; g < 2; g++) {
      const float* cg = c + 8 * g;
      w[g] = pack_e2m1x8(__fmul_rn(cg[0], k), __fmul_rn(cg[1], k), __fmul_rn(cg[2], k), __fmul_rn(cg[3], k),
                         __fmul_rn(cg[4], k), __fmul_rn(cg[5], k), __fmul_rn(cg[6], k), __fmul_rn(cg[7], k));
    }
    if (sc == 0u) w[0] = w[1] = 0u;
    if (real) crow[b] = make_uint2(w[0], w[1]);
    sw[b / 4] |= sc << (8 * (b % 4));
  }
  uint32_t* atom = T.scales + (bh * p.NT + t) * (2 * kSfAtomBytes / 4);
  atom[(r % 32) * 4 + (r / 32)] = sw[0];
  atom[kSfAtomBytes / 4 + (r % 32) * 4 + (r / 32)] = sw[1];
}

// NVFP4 V tile: warp kb takes tokens 32kb .. 32kb+31 (two 16-token blocks);
// lane l owns channels 2l, 2l+1, 64+2l, 65+2l.
__device__ __forceinline__ void quantize_v_tile_nv(const uint8_t* tile, int kb, int lane, int64_t bh, int64_t t,
                                                   const QParams& p, const QTensor& T, uint32_t empty_bar) {
  uint32_t w[2][kBlock];
#pragma unroll
  for (int i = 0; i < kBlock; i++) {
    const int row = kb * kBlock + i;
    const int off = row * 128 + ((((lane >> 2) ^ (row & 7))) << 4) + ((lane & 3) << 2);
    w[0][i] = *reinterpret_cast<const uint32_t*>(tile + off);
    w[1][i] = *reinterpret_cast<const uint32_t*>(tile + kQHalfBytes + off);
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(empty_bar);
  const float et = nv_encode(T.amax);
  const int64_t tok0 = t * kTile + kb * kBlock;
  uint8_t* sbytes = reinterpret_cast<uint8_t*>(T.scales + (bh * p.NT + t) * (2 * kSfAtomBytes / 4)) +
                    (kb / 2) * kSfAtomBytes;
#pragma unroll
  for (int h = 0; h < 2; h++) {
    uint32_t cw[2][4];
    const int c0 = 64 * h + 2 * lane;
#pragma unroll
    for (int j = 0; j < 2; j++) {  // tokens 16j .. 16j+15 of the warp's 32
      uint32_t mw = w[h][16 * j] & 0x7FFF7FFFu;
#pragma unroll
      for (int i = 1; i < 16; i++) {
        const uint32_t a = w[h][16 * j + i] & 0x7FFF7FFFu;
        asm("max.bf16x2 %0, %0, %1;" : "+r"(mw) : "r"(a));
      }
      float m2[2];
      bf16x2_to_f32(mw, m2[0], m2[1]);
      float k2[2];
      uint32_t sc[2];
#pragma unroll
      for (int q = 0; q < 2; q++) sc[q] = nv_block_scale(m2[q], et, &k2[q]);
#pragma unroll
      for (int g = 0; g < 2; g++) {
        float q0[8], q1[8];
#pragma unroll
        for (int i = 0; i < 8; i++) {
          float lo, hi;
          bf16x2_to_f32(w[h][16 * j + 8 * g + i], lo, hi);
          q0[i] = __fmul_rn(lo, k2[0]);
          q1[i] = __fmul_rn(hi, k2[1]);
        }
        cw[0][2 * j + g] = sc[0] ? pack_e2m1x8(q0[0], q0[1], q0[2], q0[3], q0[4], q0[5], q0[6], q0[7]) : 0u;
        cw[1][2 * j + g] = sc[1] ? pack_e2m1x8(q1[0], q1[1], q1[2], q1[3], q1[4], q1[5], q1[6], q1[7]) : 0u;
      }
      // block 2*kb + j of the tile -> atom kb/2, byte 2*(kb%2) + j
#pragma unroll
      for (int q = 0; q < 2; q++) {
        const int c = c0 + q;
        sbytes[(c % 32) * 16 + (c / 32) * 4 + 2 * (kb % 2) + j] = static_cast<uint8_t>(sc[q]);
      }
    }
    if (tok0 < p.N) {
#pragma unroll
      for (int q = 0; q < 2; q++)
        *reinterpret_cast<uint4*>(T.codes + (bh * kD + c0 + q) * p.row_bytes + tok0 / 2) =
            make_uint4(cw[q][0], cw[q][1], cw[q][2], cw[q][3]);
    }
  }
}

// max |x| of a bf16 tensor into *amax_bits (zeroed before the launch): the
// bits of a nonnegative binary32 order like the values.
__global__ void __launch_bounds__(256) amax_kernel(const uint4* __restrict__ x, int64_t nvec,
                                                   uint32_t* __restrict__ amax_bits) {
  uint32_t m = 0u;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; i < nvec;
       i += static_cast<int64_t>(gridDim.x) * 256) {
    const uint4 u = __ldg(x + i);
    const uint32_t a[4] = {u.x & 0x7FFF7FFFu, u.y & 0x7FFF7FFFu, u.z & 0x7FFF7FFFu, u.w & 0x7FFF7FFFu};
#pragma unroll
    for (int j = 0; j < 4; j++) asm("max.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(a[j]));
  }
  float lo, hi;
  bf16x2_to_f32(m, lo, hi);
  float f = fmaxf(lo, hi);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) f = fmaxf(f, __shfl_xor_sync(0xffffffffu, f, d));
  if ((threadIdx.x & 31) == 0 && f > 0.0f) atomicMax(amax_bits, __float_as_uint(f));
}

__device__ __forceinline__ void quantize_qk_tile(const uint8_t* tile, int r, int64_t bh, int64_t t, const QParams& p,
                                                 const QTensor& T, uint32_t empty_bar) {
  float z[kD];
#pragma unroll
  for (int c = 0; c < kD / 8; c++) {
    const uint4 raw = *reinterpret_cast<const uint4*>(tile + (c >> 3) * kQHalfBytes + r * 128 +
                                                      (((c & 7) ^ (r & 7)) << 4));
    bf16x2_to_f32(raw.x, z[8 * c + 0], z[8 * c + 1]);
    bf16x2_to_f32(raw.y, z[8 * c + 2], z[8 * c + 3]);
    bf16x2_to_f32(raw.z, z[8 * c + 4], z[8 * c + 5]);
    bf16x2_to_f32(raw.w, z[8 * c + 6], z[8 * c + 7]);
  }
  // the tile is in registers: hand the stage back to the producer
  __syncwarp();
  if ((r & 31) == 0) mbar_arrive(empty_bar);
  if (T.rotate) {
#pragma unroll
    for (int i = 0; i < kD; i += 2) bfly(z[i], z[i + 1]);  // h = 1
#pragma unroll
    for (int h = 2; h < kD; h *= 2) {
#pragma unroll
      for (int i = 0; i < kD; i += 2)
        if ((i & h) == 0) bfly2(z[i], z[i + 1], z[i + h], z[i + h + 1]);
    }
    const float2 rs = make_float2(kRotScale, kRotScale);
#pragma unroll
    for (int i = 0; i < kD; i += 2) {
      const float2 v = __fmul2_rn(make_float2(z[i], z[i + 1]), rs);
      z[i] = v.x;
      z[i + 1] = v.y;
    }
  }
  const int64_t n = t * kTile + r;
  const bool real = n < p.N;
  uint4* crow = reinterpret_cast<uint4*>(T.codes) + (bh * p.N + n) * (kD / 32);
  uint32_t sw = 0;
#pragma unroll
  for (int k = 0; k < kD / kBlock; k++) {
    const float* c = z + kBlock * k;
    const float m = absmax32(c);
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    uint32_t sbyte = 127;
    if (m > 0.0f) {
      const int e = block_exponent(m, T.rule);
      const float2 inv = make_float2(pow2_neg(e), pow2_neg(e));
#pragma unroll
      for (int g = 0; g < 4; g++) {
        const float* cg = c + 8 * g;
        const float2 a = __fmul2_rn(make_float2(cg[0], cg[1]), inv), b = __fmul2_rn(make_float2(cg[2], cg[3]), inv);
        const float2 cc = __fmul2_rn(make_float2(cg[4], cg[5]), inv), d = __fmul2_rn(make_float2(cg[6], cg[7]), inv);
        w[g] = pack_e2m1x8(a.x, a.y, b.x, b.y, cc.x, cc.y, d.x, d.y);
      }
      sbyte = static_cast<uint32_t>(e + 127);
    }
    if (real) crow[k] = make_uint4(w[0], w[1], w[2], w[3]);
    sw |= sbyte << (8 * k);
  }
  // padding rows (n >= N) read zeros and store byte 127 in every block
  T.scales[(bh * p.NT + t) * (kSfAtomBytes / 4) + (r % 32) * 4 + (r / 32)] = sw;
}

__device__ __forceinline__ void quantize_v_tile(const uint8_t* tile, int kb, int lane, int64_t bh, int64_t t,
                                                const QParams& p, const QTensor& T, uint32_t empty_bar) {
  uint32_t w[2][kBlock];
#pragma unroll
  for (int i = 0; i < kBlock; i++) {
    const int row = kb * kBlock + i;
    const int off = row * 128 + ((((lane >> 2) ^ (row & 7))) << 4) + ((lane & 3) << 2);
    w[0][i] = *reinterpret_cast<const uint32_t*>(tile + off);
    w[1][i] = *reinterpret_cast<const uint32_t*>(tile + kQHalfBytes + off);
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(empty_bar);
  const int64_t tok0 = t * kTile + kb * kBlock;
  uint8_t* sbytes = reinterpret_cast<uint8_t*>(T.scales + (bh * p.NT + t) * (kSfAtomBytes / 4));
#pragma unroll
  for (int h = 0; h < 2; h++) {
    // |.| maxima of both channels of the word at once: bf16 max is exact
    uint32_t mw = w[h][0] & 0x7FFF7FFFu;
#pragma unroll
    for (int i = 1; i < kBlock; i++) {
      const uint32_t a = w[h][i] & 0x7FFF7FFFu;
      asm("max.bf16x2 %0, %0, %1;" : "+r"(mw) : "r"(a));
    }
    float m2[2];
    bf16x2_to_f32(mw, m2[0], m2[1]);
    uint32_t sb[2];
    float inv[2];
#pragma unroll
    for (int q = 0; q < 2; q++) {
      const bool nz = m2[q] > 0.0f;
      const int e = nz ? block_exponent(m2[q], T.rule) : 0;
      sb[q] = nz ? static_cast<uint32_t>(e + 127) : 127u;
      inv[q] = nz ? pow2_neg(e) : 0.0f;
    }
    uint32_t cw[2][4];
    const float2 inv2 = make_float2(inv[0], inv[1]);
#pragma unroll
    for (int g = 0; g < 4; g++) {
      float q0[8], q1[8];
#pragma unroll
      for (int i = 0; i < 8; i++) {
        float lo, hi;
        bf16x2_to_f32(w[h][8 * g + i], lo, hi);
        const float2 q = __fmul2_rn(make_float2(lo, hi), inv2);
        q0[i] = q.x;
        q1[i] = q.y;
      }
      cw[0][g] = pack_e2m1x8(q0[0], q0[1], q0[2], q0[3], q0[4], q0[5], q0[6], q0[7]);
      cw[1][g] = pack_e2m1x8(q1[0], q1[1], q1[2], q1[3], q1[4], q1[5], q1[6], q1[7]);
    }
    const int c0 = 64 * h + 2 * lane;
    if (tok0 < p.N) {  // block holds at least one real token; it lies inside Npad
#pragma unroll
      for (int q = 0; q < 2; q++)
        *reinterpret_cast<uint4*>(T.codes + (bh * kD + c0 + q) * p.row_bytes + tok0 / 2) =
            make_uint4(cw[q][0], cw[q][1], cw[q][2], cw[q][3]);
    }
    // scale byte of row c, block kb -> (c%32)*16 + (c/32)*4 + kb
#pragma unroll
    for (int q = 0; q < 2; q++) {
      const int c = c0 + q;
      sbytes[(c % 32) * 16 + (c / 32) * 4 + kb] = static_cast<uint8_t>(sb[q]);
    }
  }
}

__global__ void __launch_bounds__(kQThreads, kQMinBlocks)
    quantize_tiles_kernel(const __grid_constant__ CUtensorMap m0, const __grid_constant__ CUtensorMap m1,
                          const __grid_constant__ CUtensorMap m2, const __grid_constant__ QParams p) {
  extern __shared__ __align__(1024) uint8_t qsmem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(qsmem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kQStages * kQStageBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kQStages);
  const uint32_t sb = smem_u32(smem);
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto empty = [&](int s) { return smem_u32(&bars[kQStages + s]); };
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const bool leader = threadIdx.x == 0;
  const int nt = p.ntensors;
  // unit g (global) -> tensor g % nt, tile g / nt = (head, 128-token tile)
  auto issue = [&](uint32_t j) {  // local unit j of this CTA into stage j % kQStages
    const int64_t g = blockIdx.x + static_cast<int64_t>(j) * gridDim.x;
    const int s = j % kQStages;
    const int ti = static_cast<int>(g % nt);
    const int64_t tile = g / nt;
    const int bh = static_cast<int>(tile / p.NT);
    const int t = static_cast<int>(tile - static_cast<int64_t>(bh) * p.NT);
    const CUtensorMap* m = ti == 0 ? &m0 : (ti == 1 ? &m1 : &m2);
    mbar_arrive_expect_tx(full(s), kQStageBytes);
    tma_load_3d(sb + s * kQStageBytes, m, full(s), 0, t * kTile, bh);
    tma_load_3d(sb + s * kQStageBytes + kQHalfBytes, m, full(s), 64, t * kTile, bh);
  };
  const uint32_t nunits =
      p.units > blockIdx.x ? static_cast<uint32_t>((p.units - blockIdx.x + gridDim.x - 1) / gridDim.x) : 0u;
  uint32_t issued = 0;
  if (leader) {
    *abort_flag = 0;
    for (int s = 0; s < kQStages; s++) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), kQConsumers / 32);
    }
    fence_mbar_init();
    prefetch_tmap(&m0);
    if (nt > 1) prefetch_tmap(&m1);
    if (nt > 2) prefetch_tmap(&m2);
    for (; issued < nunits && issued < static_cast<uint32_t>(kQStages); issued++) issue(issued);
  }
  __syncthreads();
  for (uint32_t i = 0; i < nunits; i++) {
    // the leader refills the stage that unit i-1 used with unit i-1+kQStages,
    // once all four warps have read unit i-1 into registers
    if (leader && i >= 1 && issued < nunits) {
      const uint32_t prev = i - 1;
      if (!mbar_wait(empty(prev % kQStages), (prev / kQStages) & 1, abort_flag)) {
        record_error(p.status, 4, const_cast<int*>(abort_flag));
      } else {
        issue(issued);
        issued++;
      }
    }
    const int s = i % kQStages;
    if (!mbar_wait(full(s), (i / kQStages) & 1, abort_flag)) {
      record_error(p.status, 4, const_cast<int*>(abort_flag));
      break;
    }
    const int64_t g = blockIdx.x + static_cast<int64_t>(i) * gridDim.x;
    const int ti = static_cast<int>(g % nt);
    const int64_t tile = g / nt;
    const int64_t bh = tile / p.NT;
    const int64_t t = tile - bh * p.NT;
    // a copy picked by value: a run-time index into the parameter array would go through local memory
    const QTensor T = ti == 0 ? p.t[0] : (ti == 1 ? p.t[1] : p.t[2]);
    const uint8_t* st = smem + s * kQStageBytes;
    if (T.nv) {
      if (T.is_v)
        quantize_v_tile_nv(st, warp, lane, bh, t, p, T, empty(s));
      else
        quantize_qk_tile_nv(st, threadIdx.x, bh, t, p, T, empty(s));
    } else if (T.is_v) {
      quantize_v_tile(st, warp, lane, bh, t, p, T, empty(s));
    } else {
      quantize_qk_tile(st, threadIdx.x, bh, t, p, T, empty(s));
    }
  }
  // after an abort, every copy the leader issued must land before the CTA exits
  if (leader && *abort_flag) {
    for (uint32_t j = 0; j < issued; j++) mbar_wait(full(j % kQStages), (j / kQStages) & 1, abort_flag);
  }
}

// ----------------------------------------------------- fused Q/K/V by role
// The one-launch quantizer of a forward (mxattn_quantize_qkv: Q and K rotated,
// V not, MXFP4) with the work split by role inside one CTA per SM: warpgroups
// 0 and 1 take the Q and K tiles (one thread per token, 200 registers), and
// warpgroup 2 the V tiles (104 registers; setmaxnreg moves the difference:
// 2 * 128 * 200 + 128 * 104 = 384 * 168, the launch allocation).
// Each warpgroup has its own two-stage TMA ring and leader thread. Three warps
// then share every SM sub-partition, and the V tiles' light, memory-bound
// work runs beside the rotation's ALU work instead of taking turns with it.
// Same per-tile code (quantize_qk_tile, quantize_v_tile), so the same bytes.
constexpr int kRThreads = 384;
constexpr int kRStages = 2;
constexpr uint32_t kRRingBytes = kRStages * kQStageBytes;                // 64 KB per warpgroup
constexpr uint32_t kRSmemBytes = 3 * kRRingBytes + 3 * 2 * kRStages * 8 + 16 + 1024;

__global__ void __launch_bounds__(kRThreads, 1)
    quantize_qkv_roles_kernel(const __grid_constant__ CUtensorMap m0, const __grid_constant__ CUtensorMap m1,
                              const __grid_constant__ CUtensorMap m2, const __grid_constant__ QParams p) {
  extern __shared__ __align__(1024) uint8_t qsmem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(qsmem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 3 * kRRingBytes);  // [3 rings][full, empty][stages]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 3 * 2 * kRStages);
  const int wg = threadIdx.x / 128;     // 0, 1: Q/K tiles; 2: V tiles
  const int t128 = threadIdx.x % 128;   // thread within the warpgroup
  const int wwarp = t128 / 32, lane = t128 % 32;
  const bool leader = t128 == 0;
  const uint32_t ring = smem_u32(smem + wg * kRRingBytes);
  auto full = [&](int s) { return smem_u32(&bars[(wg * 2 + 0) * kRStages + s]); };
  auto empty = [&](int s) { return smem_u32(&bars[(wg * 2 + 1) * kRStages + s]); };
  const int64_t G = gridDim.x, c = blockIdx.x;
  const int64_t U = p.BH * p.NT;  // tiles per tensor
  // this warpgroup's units: Q/K unit u (tensor u % 2, tile u / 2) for u = c + i*G,
  // i = wg, wg + 2, ...; V tile c + i*G for i = 0, 1, ...
  const int64_t first = wg < 2 ? c + wg * G : c;
  const int64_t step = wg < 2 ? 2 * G : G;
  const int64_t total = wg < 2 ? 2 * U : U;
  const uint32_t nunits = first < total ? static_cast<uint32_t>((total - first + step - 1) / step) : 0u;
  auto issue = [&](uint32_t j) {
    const int64_t u = first + static_cast<int64_t>(j) * step;
    const int ti = wg < 2 ? static_cast<int>(u % 2) : 2;
    const int64_t tile = wg < 2 ? u / 2 : u;
    const int bh = static_cast<int>(tile / p.NT);
    const int t = static_cast<int>(tile - static_cast<int64_t>(bh) * p.NT);
    const CUtensorMap* m = ti == 0 ? &m0 : (ti == 1 ? &m1 : &m2);
    const int s = j % kRStages;
    mbar_arrive_expect_tx(full(s), kQStageBytes);
    tma_load_3d(ring + s * kQStageBytes, m, full(s), 0, t * kTile, bh);
    tma_load_3d(ring + s * kQStageBytes + kQHalfBytes, m, full(s), 64, t * kTile, bh);
  };
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int r = 0; r < 3; r++)
      for (int s = 0; s < kRStages; s++) {
        mbar_init(smem_u32(&bars[(r * 2 + 0) * kRStages + s]), 1);
        mbar_init(smem_u32(&bars[(r * 2 + 1) * kRStages + s]), 4);
      }
    fence_mbar_init();
  }
  __syncthreads();
  // One warpgroup's loop: the leader keeps kRStages units in flight; unit i-1's
  // stage is refilled with unit i-1+kRStages once the warpgroup's four warps
  // have read unit i-1 into registers.
  auto run = [&](auto&& quantize_unit) {
    uint32_t issued = 0;
    if (leader) {
      prefetch_tmap(wg == 2 ? &m2 : (wg == 0 ? &m0 : &m1));
      for (; issued < nunits && issued < static_cast<uint32_t>(kRStages); issued++) issue(issued);
    }
    for (uint32_t i = 0; i < nunits; i++) {
      if (leader && i >= 1 && issued < nunits) {
        const uint32_t prev = i - 1;
        if (!mbar_wait(empty(prev % kRStages), (prev / kRStages) & 1, abort_flag)) {
          record_error(p.status, 4, const_cast<int*>(abort_flag));
        } else {
          issue(issued);
          issued++;
        }
      }
      const int s = i % kRStages;
      if (!mbar_wait(full(s), (i / kRStages) & 1, abort_flag)) {
        record_error(p.status, 4, const_cast<int*>(abort_flag));
        break;
      }
      quantize_unit(first + static_cast<int64_t>(i) * step, smem + wg * kRRingBytes + s * kQStageBytes, empty(s));
    }
    // after an abort, every copy the leader issued must land before the CTA exits
    if (leader && *abort_flag) {
      for (uint32_t j = 0; j < issued; j++) mbar_wait(full(j % kRStages), (j / kRStages) & 1, abort_flag);
    }
  };
  // each role's code sits wholly inside its own branch, after its register change
  if (wg < 2) {
    regs_inc<200>();
    run([&](int64_t u, const uint8_t* st, uint32_t eb) {
      const int64_t tile = u / 2;
      const int64_t bh = tile / p.NT;
      const QTensor T = (u % 2) == 0 ? p.t[0] : p.t[1];
      quantize_qk_tile(st, t128, bh, tile - bh * p.NT, p, T, eb);
    });
  } else {
    regs_dec<104>();
    run([&](int64_t u, const uint8_t* st, uint32_t eb) {
      const int64_t bh = u / p.NT;
      quantize_v_tile(st, wwarp, lane, bh, u - bh * p.NT, p, p.t[2], eb);
    });
  }
}

}  // namespace

void rule_threshold(int rule, double qmax, uint32_t* mant_thr, uint32_t* pow2_down) {
  const ScaleRule r = make_rule(rule, qmax);
  *mant_thr = r.mant_thr;
  *pow2_down = r.pow2_down;
}

cudaError_t launch_quantize(const QuantizeJob* jobs, int njobs, int64_t BH, int64_t N, cudaStream_t s) {
  if (njobs < 1 || njobs > 3) return cudaErrorInvalidValue;
  const int64_t NT = ceil_div(N, kTile);
  QParams p{};
  alignas(64) CUtensorMap maps[3];
  for (int j = 0; j < njobs; j++) {
    const uint64_t dims[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(N), static_cast<uint64_t>(BH)};
    const uint64_t strides[2] = {static_cast<uint64_t>(kD) * 2, static_cast<uint64_t>(N) * kD * 2};
    const uint32_t box[3] = {64, kTile, 1};
    if (!encode_tensor_map(&maps[j], 1, 3, const_cast<void*>(jobs[j].x), dims, strides, box, 128))
      return cudaErrorInvalidValue;
    p.t[j].codes = static_cast<uint8_t*>(jobs[j].codes);
    p.t[j].scales = static_cast<uint32_t*>(jobs[j].scales);
    p.t[j].rule = make_rule(jobs[j].rule, jobs[j].qmax);
    p.t[j].is_v = jobs[j].is_v;
    p.t[j].rotate = jobs[j].rotate;
    p.t[j].nv = jobs[j].amax != nullptr;
    p.t[j].amax = jobs[j].amax;
  }
  for (int j = njobs; j < 3; j++) maps[j] = maps[0];
  p.ntensors = njobs;
  p.BH = BH;
  p.N = N;
  p.NT = NT;
  p.row_bytes = ceil_div(N, kBlock) * kBlock / 2;
  p.units = njobs * BH * NT;
  p.status = device_status_ptr();
  if (p.status == nullptr) return cudaErrorInvalidDevice;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static int sms[64] = {0};
  static bool attr_set[64] = {false};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (sms[dev] == 0) {
    e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(quantize_tiles_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(quantize_qkv_roles_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  // the forward's one-launch quantizer (rotated Q and K, then V, MXFP4): the role-split kernel
  if (njobs == 3 && !p.t[0].nv && !p.t[1].nv && !p.t[2].nv && !p.t[0].is_v && !p.t[1].is_v && p.t[2].is_v) {
    const int64_t U = BH * NT;
    const int grid = static_cast<int>(U < sms[dev] ? U : sms[dev]);
    quantize_qkv_roles_kernel<<<grid, kRThreads, kRSmemBytes, s>>>(maps[0], maps[1], maps[2], p);
    return cudaGetLastError();
  }
  // NVFP4 jobs: the tensor maximum first (the encode factor needs it)
  for (int j = 0; j < njobs; j++) {
    if (jobs[j].amax == nullptr) continue;
    e = cudaMemsetAsync(jobs[j].amax, 0, sizeof(float), s);
    if (e != cudaSuccess) return e;
    const int64_t nvec = BH * N * (kD / 8);
    const int64_t blocks = ceil_div(nvec, 256);
    const int agrid = static_cast<int>(blocks < 8 * sms[dev] ? blocks : 8 * sms[dev]);
    amax_kernel<<<agrid, 256, 0, s>>>(static_cast<const uint4*>(jobs[j].x), nvec,
                                      reinterpret_cast<uint32_t*>(jobs[j].amax));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // persistent: as many CTAs per SM as registers and shared memory allow
  const int64_t want = kQMinBlocks * static_cast<int64_t>(sms[dev]);
  const int grid = static_cast<int>(p.units < want ? p.units : want);
  quantize_tiles_kernel<<<grid, kQThreads, kQSmemBytes, s>>>(maps[0], maps[1], maps[2], p);
  return cudaGetLastError();
}

cudaError_t launch_rotate_quantize_qk(const void* x, int64_t BH, int64_t N, void* codes, void* scales, int rule,
                                      double qmax, int rotate, cudaStream_t s) {
  const QuantizeJob j{x, codes, scales, rule, qmax, 0, rotate, nullptr};
  return launch_quantize(&j, 1, BH, N, s);
}

cudaError_t launch_quantize_v(const void* v, int64_t BH, int64_t N, void* codes, void* scales, int rule,
                              double qmax, cudaStream_t s) {
  const QuantizeJob j{v, codes, scales, rule, qmax, 1, 0, nullptr};
  return launch_quantize(&j, 1, BH, N, s);
}

}  // namespace mxattn
