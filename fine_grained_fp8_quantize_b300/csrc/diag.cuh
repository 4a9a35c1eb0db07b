// diag.cuh -- the accumulation-precision diagnostic: an E4M3 GEMM WITHOUT
// promotion, i.e. the tensor core accumulates the whole K in its own
// accumulator and nothing is scaled.  The pages report that limited
// accumulation precision in the tensor cores gives a maximum relative error
// near 2% for an inner dimension of 4096 ("Eliminate Deepseek Ai News For
// Good", the accumulation-precision sentence), which is why the method
// promotes every 128 K.  This kernel lets the same comparison be made on
// sm_103a: C = Aq . Bq^T over decoded codes, FP32 out.
//
// One CTA of 128 threads per 128 x 256 output tile, nothing overlapped: per
// K-block one thread loads the A and B tiles (TMA), issues four
// tcgen05.mma.kind::f8f6f4 (128x256x32) that accumulate into the same TMEM
// columns, and waits for them before the next load.  It exists to measure
// numerics, not speed.  Waits are bounded as in the GEMM.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "ptx.cuh"

namespace fp8q {

constexpr int kDiagBM = 128;
constexpr int kDiagBN = 256;
constexpr uint32_t kDiagABytes = 128 * 128;
constexpr uint32_t kDiagBBytes = 256 * 128;
constexpr uint32_t kDiagSmem = kDiagABytes + kDiagBBytes + 1024 + 64;  // + alignment slack, barriers
constexpr uint32_t kDiagIdesc = idesc_e4m3_f32(kDiagBM, kDiagBN);

// After a timed-out wait: give the operation 1 ms more to complete.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity) && globaltimer_ns() - t0 < 1000000ull) {}
}

__global__ void __launch_bounds__(128, 1)
    gemm_unpromoted_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, float* C,
                           int64_t M, int64_t N, int64_t K) {
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sa = smem_u32(smem);
  const uint32_t sb = sa + kDiagABytes;
  const uint32_t bar_load = sb + kDiagBBytes;
  const uint32_t bar_mma = bar_load + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kDiagABytes + kDiagBBytes + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kDiagABytes + kDiagBBytes + 20);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kDiagBM;
  const int64_t n0 = static_cast<int64_t>(blockIdx.y) * kDiagBN;
  const int64_t KB = K / 128;

  if (threadIdx.x == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (threadIdx.x == 0) {
    for (int64_t kb = 0; kb < KB; ++kb) {
      const uint32_t par = static_cast<uint32_t>(kb & 1);
      mbar_arrive_expect_tx(bar_load, kDiagABytes + kDiagBBytes);
      tma_load_2d(sa, &tmA, static_cast<int32_t>(kb * 128), static_cast<int32_t>(m0), bar_load);
      tma_load_2d(sb, &tmB, static_cast<int32_t>(kb * 128), static_cast<int32_t>(n0), bar_load);
      if (!mbar_wait(bar_load, par, abort_flag)) {
        drain_wait(bar_load, par);  // bounded: let the copies land before the CTA exits
        break;
      }
      tc_fence_after();
      const uint64_t adesc = smem_desc_k_sw128(sa);
      const uint64_t bdesc = smem_desc_k_sw128(sb);
#pragma unroll
      for (int k = 0; k < 4; ++k) mma_f8f6f4(tmem_base, adesc + 2u * k, bdesc + 2u * k, kDiagIdesc, (kb | k) ? 1u : 0u);
      mma_commit(bar_mma);
      // the stage is reused: wait until these MMAs have read it
      if (!mbar_wait(bar_mma, par, abort_flag)) {
        drain_wait(bar_mma, par);
        break;
      }
    }
  }
  __syncthreads();
  tc_fence_after();
  if (!*abort_flag) {
    const int64_t m = m0 + warp * 32 + lane;
    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      uint32_t p[32];
      tmem_ld_32x32b_x32(taddr + c * 32, p);
      tmem_ld_wait();
      const int64_t n = n0 + c * 32;
      if (m < M && n < N) {
        float4* out = reinterpret_cast<float4*>(C + m * N + n);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          out[j] = make_float4(__uint_as_float(p[4 * j]), __uint_as_float(p[4 * j + 1]), __uint_as_float(p[4 * j + 2]),
                               __uint_as_float(p[4 * j + 3]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 256);
  }
}

// Failure-detection self-test.  One thread waits on an mbarrier that nothing
// ever arrives on, through mbar_wait, the bounded wait every pipeline of this
// library uses.  The wait gives up after its limit (kWaitTimeoutNs), records
// FP8Q_ERR_TIMEOUT in the device status word and returns false, and the
// kernel ends normally: nothing traps, faults or hangs, and the context stays
// usable.
__global__ void selftest_wait_kernel() {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_word;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_word = 0;
    fence_mbar_init();
    (void)mbar_wait(smem_u32(&bar), 0, &abort_word);  // phase 0 never completes
  }
}

}  // namespace fp8q
