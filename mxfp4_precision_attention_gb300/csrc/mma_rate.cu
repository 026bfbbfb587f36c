// Tensor-core rate probe: back-to-back tcgen05.mma kind::mxf4.block_scale
// (M128 N256 or N128, K64, E2M1 operands in shared memory, UE8M0 scales in
// TMEM) with nothing else in the loop, one CTA per SM. It measures the dense FP4 MMA
// rate this GPU sustains, the figure the attention forward's tensor-core
// share is read against. Not part of the attention path.
//
// Operand pattern: every byte of A row r holds two copies of the E2M1 code
// (7r + 1) mod 16, every byte of B row n two copies of (11n + 5) mod 16, and
// every scale is 2^0. The 64-byte swizzle only permutes 16-byte chunks inside
// a row, so the logical matrices do not depend on it, and after `iters`
// iterations (two K64 MMAs each) CTA 0's accumulator is
// D[r][n] = 128 * iters * e2m1(a_r) * e2m1(b_n), exact in fp32 while
// |D| < 2^24.

#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace mxattn {
namespace {

constexpr int kThreads = 128;
constexpr uint32_t kM = 128, kNMax = 256;
constexpr uint32_t kRowBytes = 64;  // K = 128 E2M1 codes per row
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + kM * kRowBytes;  // 8 KB
constexpr uint32_t kOffBars = kOffB + kNMax * kRowBytes;  // + 16 KB
constexpr uint32_t kOffMisc = kOffBars + 64;
// Far more shared memory than the probe needs, so that one CTA fills an SM.
constexpr uint32_t kSmemBytes = 160 * 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColD = 0;     // 256 fp32 columns
constexpr uint32_t kColSF = 256;  // 32 columns of 2^0 scale bytes; A reads from +0, B from +8
constexpr int64_t kChunk = 256;   // iterations between commits

__device__ __forceinline__ uint32_t probe_row_word(uint32_t row, bool is_b) {
  const uint32_t c = is_b ? (11u * row + 5u) & 15u : (7u * row + 1u) & 15u;
  return (c | (c << 4)) * 0x01010101u;
}

__device__ __forceinline__ void probe_error(int* status, volatile int* abort_flag) {
  *abort_flag = 1;
  atomicCAS(status, 0, 4);
}

template <uint32_t kN>
__global__ void __launch_bounds__(kThreads, 1) mxf4_mma_rate_kernel(int64_t iters, float* d_out, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  // operands: a word at byte offset o of a K-major 64-byte-row tile belongs to row o / 64
  uint32_t* words = reinterpret_cast<uint32_t*>(smem);
  for (uint32_t i = threadIdx.x; i < (kOffBars - kOffA) / 4; i += kThreads) {
    const uint32_t o = 4 * i;
    words[i] = o < kOffB ? probe_row_word((o - kOffA) / kRowBytes, false) : probe_row_word((o - kOffB) / kRowBytes, true);
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    mbar_init(smem_u32(&bars[2]), 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

  // every scale byte of the 32 scale columns = 127 (2^0), whatever layout the MMA reads them in
  {
    uint32_t r[32];
#pragma unroll
    for (int j = 0; j < 32; j++) r[j] = 0x7F7F7F7Fu;
    tmem_st32(tmem + lane_base + kColSF, r);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (threadIdx.x == 0) {
    const uint32_t id0 = idesc_mxf4(kM, kN, 0, 0), id1 = idesc_mxf4(kM, kN, 2, 2);
    const uint64_t da = smem_desc(sb + kOffA, 16, 512, kSwizzle64B);
    const uint64_t db = smem_desc(sb + kOffB, 16, 512, kSwizzle64B);
    const uint32_t d = tmem + kColD, sfa = tmem + kColSF, sfb = tmem + kColSF + 8;
    const int64_t nchunks = (iters + kChunk - 1) / kChunk;
    bool ok = true;
    for (int64_t c = 0; c < nchunks && ok; c++) {
      // at most two chunks in flight: chunk c reuses the barrier of chunk c - 2
      if (c >= 2) ok = mbar_wait(smem_u32(&bars[c & 1]), static_cast<uint32_t>((c - 2) >> 1) & 1u, abort_flag);
      if (!ok) break;
      const int64_t i0 = c * kChunk, n = (iters - i0) < kChunk ? (iters - i0) : kChunk;
      for (int64_t j = 0; j < n; j++) {
        mma_mxf4(d, da, db, id0, sfa, sfb, (i0 + j) > 0 ? 1u : 0u);
        mma_mxf4(d, da + 2, db + 2, id1, sfa, sfb, 1u);  // K step 1: +32 bytes
      }
      tc_commit(smem_u32(&bars[c & 1]));
    }
    if (ok) {
      for (int64_t c = nchunks >= 2 ? nchunks - 2 : 0; c < nchunks && ok; c++)
        ok = mbar_wait(smem_u32(&bars[c & 1]), static_cast<uint32_t>(c >> 1) & 1u, abort_flag);
    } else {
      // a wait gave up: still let every MMA already issued finish before TMEM
      // is freed (a fresh barrier, so its first phase is the one to wait for)
      tc_commit(smem_u32(&bars[2]));
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(smem_u32(&bars[2]), 0u, 100000u) && globaltimer_ns() - t0 < kWaitTimeoutNs) {
      }
    }
    if (!ok) probe_error(status, abort_flag);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (d_out != nullptr && blockIdx.x == 0 && !*abort_flag) {
    for (uint32_t c0 = 0; c0 < kN; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(tmem + lane_base + kColD + c0, r);
      tmem_wait_ld();
      reg_fence32(r);
      float* row = d_out + static_cast<size_t>(warp * 32 + lane) * kN + c0;
#pragma unroll
      for (int j = 0; j < 32; j++) row[j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

double mxf4_mma_rate_flops(int64_t iters, int n, int ctas) {
  return static_cast<double>(ctas) * static_cast<double>(iters) * 2.0 * (2.0 * kM * n * 64.0);
}

cudaError_t launch_mxf4_mma_rate(int64_t iters, int n, float* d_out, int* ctas_out, cudaStream_t s) {
  if (n != 128 && n != 256) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {false};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    for (auto fn : {mxf4_mma_rate_kernel<128>, mxf4_mma_rate_kernel<256>}) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      if (e != cudaSuccess) return e;
    }
    attr_set[dev] = true;
  }
  *ctas_out = sms;
  if (n == 256) mxf4_mma_rate_kernel<256><<<sms, kThreads, kSmemBytes, s>>>(iters, d_out, device_status_ptr());
  else mxf4_mma_rate_kernel<128><<<sms, kThreads, kSmemBytes, s>>>(iters, d_out, device_status_ptr());
  return cudaGetLastError();
}

}  // namespace mxattn
