// BF16 fused attention forward (comparison path for the MXFP4 kernel):
// the FlashAttention-2 recurrence of "MXAttention" Eqs. (2)-(8) with BF16
// operands, FP32 accumulation in TMEM, Bc = 128 key tiles.
//
//   S_j = Q K_j^T                 tcgen05.mma kind::f16 (bf16) -> TMEM
//   P~  = exp(S_j/sqrt(d) - m)    fp32 in registers, rounded to bf16 -> smem
//   O   = diag(alpha) O + P V     tcgen05.mma kind::f16, V as MN-major B
//   l   = diag(alpha) l + P 1     a 16-column MMA against a constant ones tile,
//                                 so l sums exactly the bf16 P that enters O
//
// Queries and keys may differ in length (Nq, Nk); causal means key j is
// visible to query i iff j <= i. Same warp roles and bounded-wait discipline
// as the MXFP4 kernel.
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace mxattn {
namespace {

constexpr int kThreads = 384;
constexpr int kStages = 2;
constexpr uint32_t kHalfTile = 128 * 128;        // 64 bf16 x 128 rows (one 128B-swizzle column block)
constexpr uint32_t kTileB = 2 * kHalfTile;       // 32 KB
constexpr uint32_t kOnesBlock = 16 * 128;        // 16 rows x 64 keys of bf16 ones
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileB;
constexpr uint32_t kOffV = kOffK + kStages * kTileB;
constexpr uint32_t kOffP = kOffV + kStages * kTileB;
constexpr uint32_t kOffOnes = kOffP + kTileB;
constexpr uint32_t kOffXchg = kOffOnes + 2 * kOnesBlock;
constexpr uint32_t kOffLsum = kOffXchg + 2 * 2 * 128 * 4;
constexpr uint32_t kOffBars = kOffLsum + 128 * 4;
constexpr int kNumBars = 16;
constexpr uint32_t kOffMisc = kOffBars + kNumBars * 8;
constexpr uint32_t kSmemBytes = kOffMisc + 64 + 1024;

constexpr int kBarQFull = 0;
constexpr int kBarKFull = 1;
constexpr int kBarKEmpty = kBarKFull + kStages;
constexpr int kBarVFull = kBarKEmpty + kStages;
constexpr int kBarVEmpty = kBarVFull + kStages;
constexpr int kBarSFull = kBarVEmpty + kStages;
constexpr int kBarSEmpty = kBarSFull + 2;
constexpr int kBarPFull = kBarSEmpty + 2;
constexpr int kBarODone = kBarPFull + 1;
static_assert(kBarODone < kNumBars, "barrier space");

constexpr uint32_t kColS = 0;    // 2 x 128
constexpr uint32_t kColO = 256;  // 128
constexpr uint32_t kColL = 384;  // 16
constexpr uint32_t kTmemCols = 512;

struct Params {
  float* out;
  int* status;
  int64_t Nq, Nk;  // query and key/value lengths
  int NTq, NTk;     // their 128-row tile counts
  int causal;
  uint32_t debug_flags;
  float score_scale_log2;
  int bh_major;  // grid x walks heads and y walks query tiles (causal), else the reverse
};

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, %2, %3, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ void record_error(int* status, int code, volatile int* abort_flag) {
  *abort_flag = 1;
  atomicCAS(status, 0, code);
}

__global__ void __launch_bounds__(kThreads, 1)
    bf16_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int bh = static_cast<int>(p.bh_major ? blockIdx.x : blockIdx.y);
  const int slot = static_cast<int>(p.bh_major ? blockIdx.y : blockIdx.x);
  const int qt = p.causal ? (p.NTq - 1 - slot) : slot;  // causal: heaviest query tiles first
  // causal: key j is visible to query i iff j <= i (both counted from 0)
  const int T = p.causal ? (qt + 1 < p.NTk ? qt + 1 : p.NTk) : p.NTk;
  const int64_t Nq = p.Nq, Nk = p.Nk;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(kBarQFull), 1);
    for (int s = 0; s < kStages; s++) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarKEmpty + s), 1);
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarVEmpty + s), 1);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(bar(kBarSFull + b), 1);
      mbar_init(bar(kBarSEmpty + b), 8);
    }
    mbar_init(bar(kBarPFull), 8);
    mbar_init(bar(kBarODone), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_base_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp >= 4) {
    uint32_t* ones = reinterpret_cast<uint32_t*>(smem + kOffOnes);
    for (int i = threadIdx.x - 128; i < 2 * kOnesBlock / 4; i += 256) ones[i] = 0x3F803F80u;  // bf16 1.0
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_slot;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      mbar_arrive_expect_tx(bar(kBarQFull), kTileB);
      tma_load_3d(sb + kOffQ, &tm_q, bar(kBarQFull), 0, qt * 128, bh);
      tma_load_3d(sb + kOffQ + kHalfTile, &tm_q, bar(kBarQFull), 64, qt * 128, bh);
      int nk = 0, nv = 0;
      for (int j = 0; j < T; j++) {
        const int st = j % kStages, u = j / kStages;
        if (u > 0 && !mbar_wait(bar(kBarKEmpty + st), (u - 1) & 1, abort_flag)) {
          record_error(p.status, 4, abort_flag);
          break;
        }
        mbar_arrive_expect_tx(bar(kBarKFull + st), kTileB);
        tma_load_3d(sb + kOffK + st * kTileB, &tm_k, bar(kBarKFull + st), 0, j * 128, bh);
        tma_load_3d(sb + kOffK + st * kTileB + kHalfTile, &tm_k, bar(kBarKFull + st), 64, j * 128, bh);
        nk++;
        if (u > 0 && !mbar_wait(bar(kBarVEmpty + st), (u - 1) & 1, abort_flag)) {
          record_error(p.status, 4, abort_flag);
          break;
        }
        mbar_arrive_expect_tx(bar(kBarVFull + st), kTileB);
        tma_load_3d(sb + kOffV + st * kTileB, &tm_v, bar(kBarVFull + st), 0, j * 128, bh);
        tma_load_3d(sb + kOffV + st * kTileB + kHalfTile, &tm_v, bar(kBarVFull + st), 64, j * 128, bh);
        nv++;
      }
      for (int j = (nk > kStages ? nk - kStages : 0); j < nk; j++)
        mbar_wait(bar(kBarKFull + j % kStages), (j / kStages) & 1, abort_flag);
      for (int j = (nv > kStages ? nv - kStages : 0); j < nv; j++)
        mbar_wait(bar(kBarVFull + j % kStages), (j / kStages) & 1, abort_flag);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(128, 128, false);
      const uint32_t id_o = idesc_bf16(128, 128, true);
      const uint32_t id_l = idesc_bf16(128, 16, false);
      bool ok = mbar_wait(bar(kBarQFull), 0, abort_flag);
      auto issue_pv = [&](int t) -> bool {
        const int st = t % kStages;
        if (!mbar_wait(bar(kBarPFull), t & 1, abort_flag)) return false;
        if (!mbar_wait(bar(kBarVFull + st), (t / kStages) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t pa = sb + kOffP, va = sb + kOffV + st * kTileB, oa = sb + kOffOnes;
        for (int i = 0; i < 8; i++) {
          const uint64_t ad = smem_desc(pa + (i >> 2) * kHalfTile + (i & 3) * 32, 16, 1024, kSwizzle128B);
          mma_bf16(tmem + kColO, ad, smem_desc(va + i * 2048, kHalfTile, 1024, kSwizzle128B), id_o,
                   (t > 0 || i > 0) ? 1u : 0u);
          mma_bf16(tmem + kColL, ad, smem_desc(oa + (i >> 2) * kOnesBlock + (i & 3) * 32, 16, 1024, kSwizzle128B),
                   id_l, (t > 0 || i > 0) ? 1u : 0u);
        }
        tc_commit(bar(kBarODone));
        tc_commit(bar(kBarVEmpty + st));
        return true;
      };
      for (int j = 0; ok && j < T; j++) {
        const int st = j % kStages, s = j & 1;
        if (!mbar_wait(bar(kBarKFull + st), (j / kStages) & 1, abort_flag)) { ok = false; break; }
        if (j >= 2 && !mbar_wait(bar(kBarSEmpty + s), ((j >> 1) - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t ka = sb + kOffK + st * kTileB, qa = sb + kOffQ;
        for (int i = 0; i < 8; i++) {
          const uint32_t off = (i >> 2) * kHalfTile + (i & 3) * 32;
          mma_bf16(tmem + kColS + s * 128, smem_desc(qa + off, 16, 1024, kSwizzle128B),
                   smem_desc(ka + off, 16, 1024, kSwizzle128B), id_s, i > 0 ? 1u : 0u);
        }
        if (!((p.debug_flags & kDebugNeverArriveS) && j == 0)) tc_commit(bar(kBarSFull + s));
        tc_commit(bar(kBarKEmpty + st));
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok && !issue_pv(T - 1)) ok = false;
      if (!ok) record_error(p.status, 4, abort_flag);
    }
  } else if (warp >= 4) {
    const int h = (warp - 4) / 4;
    const int quad = warp % 4;
    const int r = quad * 32 + lane;
    const int64_t qrow = static_cast<int64_t>(qt) * 128 + r;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    float* xchg = reinterpret_cast<float*>(smem + kOffXchg);
    float* lsum = reinterpret_cast<float*>(smem + kOffLsum);
    const float C = p.score_scale_log2;
    const bool ragged = (Nk % 128) != 0;
    float m_run = -INFINITY;
    bool my_abort = false, aborted = false;
    auto wait_uniform = [&](int b, uint32_t parity) {
      bool ok = !my_abort && mbar_wait(bar(b), parity, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok && !my_abort) {
        record_error(p.status, 4, abort_flag);
        my_abort = true;
      }
    };
    for (int j = 0; j < T; j++) {
      const int s = j & 1;
      float v[64];
      float pm = 0.0f;  // this warp's half-row maximum (from the loads themselves)
      wait_uniform(kBarSFull + s, (j >> 1) & 1);
      tc_fence_after();
      if (!my_abort) {
        uint32_t r0[32], r1[32];
        float m0, m1;
        tmem_ld32_max(tl + kColS + s * 128 + 64 * h, r0, m0);
        tmem_ld32_max(tl + kColS + s * 128 + 64 * h + 32, r1, m1);
        tmem_wait_ld();
        reg_fence32(r0);
        reg_fence32(r1);
        uint32_t u0 = __float_as_uint(m0), u1 = __float_as_uint(m1);
        reg_fence1(u0);
        reg_fence1(u1);
        pm = fmaxf(__uint_as_float(u0), __uint_as_float(u1));
#pragma unroll
        for (int i = 0; i < 32; i++) {
          v[i] = __uint_as_float(r0[i]);
          v[32 + i] = __uint_as_float(r1[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 64; i++) v[i] = 0.0f;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarSEmpty + s));
      const int64_t key0 = static_cast<int64_t>(j) * 128 + 64 * h;
      if (j == T - 1 && (p.causal || ragged)) {
        // the last tile's masked keys are -inf in v only: its maximum comes from v
#pragma unroll
        for (int i = 0; i < 64; i++) {
          const int64_t key = key0 + i;
          if (!(key < Nk && (!p.causal || key <= qrow))) v[i] = -INFINITY;
        }
        pm = v[0];
#pragma unroll
        for (int i = 1; i < 63; i += 2) pm = fmax3(pm, v[i], v[i + 1]);
        pm = fmaxf(pm, v[63]);
      }
      xchg[(s * 2 + h) * 128 + r] = pm;
      aborted = bar_red_or(1, 256, my_abort || *abort_flag);
      if (aborted) break;
      const float other = xchg[(s * 2 + (1 - h)) * 128 + r];
      const float m_new = fmax3(m_run, pm, other);
      const float mc = m_new * C;
      uint32_t packed[32];
      const float2 c2 = make_float2(C, C), nmc2 = make_float2(-mc, -mc);
#pragma unroll
      for (int i = 0; i < 32; i++) {
        const float2 x = __ffma2_rn(make_float2(v[2 * i], v[2 * i + 1]), c2, nmc2);
        packed[i] = pack_bf16x2(ex2_approx(x.x), ex2_approx(x.y));
      }
      const float alpha = (j == 0) ? 0.0f : ex2_approx((m_run - m_new) * C);
      if (j >= 1) {
        // PV_{j-1} done: P buffer free and O ready for rescaling
        wait_uniform(kBarODone, (j - 1) & 1);
        tc_fence_after();
      }
      {
        uint8_t* prow = smem + kOffP + h * kHalfTile + r * 128;
        const int x = r & 7;
#pragma unroll
        for (int c = 0; c < 8; c++)
          *reinterpret_cast<uint4*>(prow + ((c ^ x) << 4)) =
              make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
      }
      fence_proxy_async_smem();
      if (j >= 1 && !my_abort && __any_sync(0xffffffffu, alpha != 1.0f)) {
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int c = 0; c < 2; c++) {
          uint32_t o[32];
          tmem_ld32(tl + kColO + 64 * h + 32 * c, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 x = __fmul2_rn(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), a2);
            o[i] = __float_as_uint(x.x);
            o[i + 1] = __float_as_uint(x.y);
          }
          tmem_st32(tl + kColO + 64 * h + 32 * c, o);
        }
        if (h == 1) {
          const uint32_t l = tmem_ld1(tl + kColL);
          tmem_wait_ld();
          tmem_st1(tl + kColL, __float_as_uint(__uint_as_float(l) * alpha));
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull));
      m_run = m_new;
    }
    if (!aborted) wait_uniform(kBarODone, (T - 1) & 1);
    tc_fence_after();
    if (h == 1) {
      float l = 0.0f;
      if (!my_abort && !aborted) {
        l = __uint_as_float(tmem_ld1(tl + kColL));
        tmem_wait_ld();
      }
      lsum[r] = l;
    }
    named_bar_sync(2, 256);
    const float inv_l = 1.0f / lsum[r];
    if (!my_abort && !aborted) {
      float4* dst = reinterpret_cast<float4*>(p.out + (static_cast<int64_t>(bh) * Nq + qrow) * kD + 64 * h);
      for (int c = 0; c < 2; c++) {
        uint32_t rr[32];
        tmem_ld32(tl + kColO + 64 * h + 32 * c, rr);  // warp-wide; rows past Nq load but do not store
        tmem_wait_ld();
        if (qrow < Nq) {
#pragma unroll
          for (int i = 0; i < 8; i++)
            dst[8 * c + i] = make_float4(__uint_as_float(rr[4 * i]) * inv_l, __uint_as_float(rr[4 * i + 1]) * inv_l,
                                         __uint_as_float(rr[4 * i + 2]) * inv_l,
                                         __uint_as_float(rr[4 * i + 3]) * inv_l);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_bf16_forward(const Bf16FwdArgs& a, cudaStream_t s) {
  const int64_t Nq = a.Nq, Nk = a.Nk, BH = a.BH;
  const int64_t NTq = ceil_div(Nq, 128), NTk = ceil_div(Nk, 128);
  alignas(64) CUtensorMap tq, tk, tv;
  const uint64_t dq[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(Nq), static_cast<uint64_t>(BH)};
  const uint64_t sq[2] = {kD * 2, static_cast<uint64_t>(Nq) * kD * 2};
  const uint64_t dk[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(Nk), static_cast<uint64_t>(BH)};
  const uint64_t sk[2] = {kD * 2, static_cast<uint64_t>(Nk) * kD * 2};
  const uint32_t box[3] = {64, 128, 1};
  if (!encode_tensor_map(&tq, 1, 3, const_cast<void*>(a.q), dq, sq, box, 128)) return cudaErrorInvalidValue;
  if (!encode_tensor_map(&tk, 1, 3, const_cast<void*>(a.k), dk, sk, box, 128)) return cudaErrorInvalidValue;
  if (!encode_tensor_map(&tv, 1, 3, const_cast<void*>(a.v), dk, sk, box, 128)) return cudaErrorInvalidValue;
  Params p;
  p.out = a.out;
  p.status = device_status_ptr();
  p.Nq = Nq;
  p.Nk = Nk;
  p.NTq = static_cast<int>(NTq);
  p.NTk = static_cast<int>(NTk);
  p.causal = a.causal;
  p.debug_flags = a.debug_flags;
  p.score_scale_log2 = 1.4426950408889634f / 11.313708498984761f;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {false};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(bf16_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  // causal: heads on x so that every head's longest query tile starts first
  p.bh_major = (a.causal && NTq <= 65535) ? 1 : 0;
  dim3 grid = p.bh_major ? dim3(static_cast<unsigned>(BH), static_cast<unsigned>(NTq))
                         : dim3(static_cast<unsigned>(NTq), static_cast<unsigned>(BH));
  bf16_fwd_kernel<<<grid, kThreads, kSmemBytes, s>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace mxattn
