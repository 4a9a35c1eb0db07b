// mx.cuh -- the MX (microscaling) variant for sm_103a: E4M3 codes in 1x32
// groups with power-of-two E8M0 scales, and a GEMM whose tensor cores apply
// those scales themselves (tcgen05.mma.kind::mxf8f6f4.block_scale).
//
// The pages note that the fine-grained 1x128 / 128x128 strategy follows the
// microscaling formats, and that Blackwell tensor cores support them with
// smaller groups ("Deepseek Ai News Expert Interview", the DualPipe /
// microscaling paragraph).  The conversion is the one the MX formats define:
//   shared exponent e = floor(log2(amax)) - 8 (8: the exponent of E4M3's top
//   binade, 448 = 1.75 * 2^8), clamped to [-127, 127], 0 -> -127;
//   scale byte (E8M0) = e + 127;  code = E4M3_rn_satfinite(x * 2^-e).
// For a normal FP32 amax with biased exponent b, floor(log2(amax)) = b - 127,
// so the scale byte is max(b - 8, 0) (zero and subnormal amax give 0), and
// 2^-e is the normal float with biased exponent 254 - byte.  x * 2^-e is
// exact (or the correctly rounded subnormal), so it equals x / 2^e.
//
// Scale layout (both operands, rows x K):  s[K/128][ceil(rows/128)][512]
// bytes; the 512-byte chunk of row tile rt and K-block kt holds the scale of
// row r (0..127) and 32-group c (0..3) at byte (r % 32) * 16 + (r / 32) * 4
// + c.  A chunk is the 32-row x 16-byte matrix that tcgen05.cp's 32x128b
// shape moves into TMEM (replicated to the four lane quarters), which is
// where the block-scaled MMA reads its scale factors; chunks of one K-block
// are contiguous, so the B scales of a 256-row tile are one 1 KB copy.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "ptx.cuh"

namespace fp8q {

// ---------------------------------------------------------------------------
// Quantizer: 1x32 groups along K, E8M0 scales (FP32 input; BF16 input runs
// the TMA-fed quant_rc_kernel in its MX mode, same arithmetic)
// ---------------------------------------------------------------------------
// Work unit: a slab of 16 rows x 128 columns (one eighth of a 128 x 128
// tile), one warp per slab, slabs striped over all warps of a persistent
// grid; warps never wait for each other.  Per step a warp reads two slab rows
// (lanes 0-15 the first, 16-31 the second), each lane 8 consecutive
// elements, so one 32-element group spans 4 lanes and its amax is two
// shuffles.  All eight steps' loads are issued before any arithmetic.  Codes
// leave as 8-byte stores (a half-warp writes one 128-byte row segment).  The
// four scale bytes of one row in one K-block are adjacent in the tiled
// layout, so they leave as one 4-byte store.
constexpr int kMxQuantThreads = 256;

__device__ __forceinline__ uint32_t mx_scale_byte(float amax) {
  const int b = static_cast<int>(__float_as_uint(amax) >> 23);  // amax >= 0: biased exponent
  return static_cast<uint32_t>(b > 8 ? b - 8 : 0);
}

template <bool kF32>
__global__ void __launch_bounds__(kMxQuantThreads)
    quant_mx_kernel(const void* __restrict__ x, int64_t rows, int64_t K, uint8_t* __restrict__ q,
                    uint8_t* __restrict__ s, int64_t num_slabs) {
  const int lane = threadIdx.x & 31;
  const int64_t KT = K >> 7;
  const int64_t RT = (rows + 127) >> 7;
  const int half = lane >> 4;   // which of the two rows of a step
  const int col8 = lane & 15;   // 8-column slot within the row
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kMxQuantThreads / 32);

  for (int64_t sl = static_cast<int64_t>(blockIdx.x) * (kMxQuantThreads / 32) + (threadIdx.x >> 5); sl < num_slabs;
       sl += warps) {
    const int64_t t = sl >> 3;        // tile
    const int w = static_cast<int>(sl & 7);  // slab within the tile: rows 16w .. 16w+15
    const int64_t rt = t / KT;
    const int64_t kt = t - rt * KT;
    const int64_t col = kt * 128 + col8 * 8;
    constexpr int kWords = kF32 ? 2 : 1;  // 16-byte words per lane per row
    uint4 v[8][kWords];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t m = rt * 128 + w * 16 + 2 * i + half;
      if (m < rows) {
        if constexpr (kF32) {
          const uint4* p = reinterpret_cast<const uint4*>(static_cast<const float*>(x) + m * K + col);
          v[i][0] = __ldg(p);
          v[i][kWords - 1] = __ldg(p + 1);
        } else {
          v[i][0] = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + m * K + col));
        }
      } else {
#pragma unroll
        for (int j = 0; j < kWords; ++j) v[i][j] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = w * 16 + 2 * i + half;  // tile-local row
      const int64_t m = rt * 128 + r;
      float e[8];
      float amax;
      if constexpr (kF32) {
        e[0] = __uint_as_float(v[i][0].x); e[1] = __uint_as_float(v[i][0].y);
        e[2] = __uint_as_float(v[i][0].z); e[3] = __uint_as_float(v[i][0].w);
        e[4] = __uint_as_float(v[i][kWords - 1].x); e[5] = __uint_as_float(v[i][kWords - 1].y);
        e[6] = __uint_as_float(v[i][kWords - 1].z); e[7] = __uint_as_float(v[i][kWords - 1].w);
        amax = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(e[j]));
      } else {
        // packed BF16 |x| max (exact), then widen
        const uint4 u = v[i][0];
        const __nv_bfloat162 a2 = __hmax2(__hmax2(__habs2(bf2_of(u.x)), __habs2(bf2_of(u.y))),
                                          __hmax2(__habs2(bf2_of(u.z)), __habs2(bf2_of(u.w))));
        const uint32_t ab = u32_of(a2);
        amax = fmaxf(bf16lo_to_f32(ab), bf16hi_to_f32(ab));
        e[0] = bf16lo_to_f32(u.x); e[1] = bf16hi_to_f32(u.x);
        e[2] = bf16lo_to_f32(u.y); e[3] = bf16hi_to_f32(u.y);
        e[4] = bf16lo_to_f32(u.z); e[5] = bf16hi_to_f32(u.z);
        e[6] = bf16lo_to_f32(u.w); e[7] = bf16hi_to_f32(u.w);
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      const uint32_t byte = mx_scale_byte(amax);
      const float inv = __uint_as_float((254u - byte) << 23);  // 2^-(byte - 127), a normal float
      // the row's four scale bytes (groups 0..3 sit on lanes 0, 4, 8, 12 of its half)
      const int base = lane & 16;
      const uint32_t word = __shfl_sync(0xffffffffu, byte, base) | (__shfl_sync(0xffffffffu, byte, base + 4) << 8) |
                            (__shfl_sync(0xffffffffu, byte, base + 8) << 16) |
                            (__shfl_sync(0xffffffffu, byte, base + 12) << 24);
      if (m < rows) {
        const uint2 c = make_uint2(cvt_e4m3x4(e[0] * inv, e[1] * inv, e[2] * inv, e[3] * inv),
                                   cvt_e4m3x4(e[4] * inv, e[5] * inv, e[6] * inv, e[7] * inv));
        *reinterpret_cast<uint2*>(q + m * K + col) = c;
      }
      if (col8 == 0)  // rows past the end get scale 1 (byte 127): defined, never read into C
        *reinterpret_cast<uint32_t*>(s + (kt * RT + rt) * 512 + (r & 31) * 16 + (r >> 5) * 4) =
            m < rows ? word : 0x7F7F7F7Fu;
    }
  }
}

// ---------------------------------------------------------------------------
// GEMM: C = (A * 2^sA) (B * 2^sB)^T with the scales applied by the tensor core
// ---------------------------------------------------------------------------
// Persistent, warp-specialised, one CTA of 320 threads per SM, 128 x 256
// output tiles, K-blocks of 128:
//   warp 0       TMA producer: per K-block one 128x128 A tile and one
//                256x128 B tile (128-byte swizzle) plus the K-block's scale
//                chunks (A 512 bytes, B 1 KB) into a 4-stage ring.
//   warp 1       TMEM owner and MMA issuer: per K-block it copies the
//                scale chunks into the stage's TMEM scale columns
//                (tcgen05.cp) and issues four block-scaled MMAs
//                (128x256x32, scale byte k of each column for step k) that
//                accumulate the whole K of the tile in one TMEM accumulator.
//   warps 2-9    epilogue: each thread reads one row x 128 columns of the
//                finished accumulator, frees it for the next tile's MMAs,
//                and stores BF16 (RNE) or FP32 through TMA.
// TMEM: accumulator in columns 0-255; stage s's scale factors in columns
// 256 + 32 s (A: 4 columns, B: 8 columns at +16).  A stage's scale columns
// are rewritten only after the MMAs that read them have completed: the
// producer refills a stage after the MMAs' commit frees it.
// Warps 0 and 1 run their loops as whole warps and issue from one elected
// lane (elect.sync): the operands stay warp-uniform, which makes each issued
// operation several times cheaper for the issuing thread than the same loop
// run by lane 0 alone (measured: ~600 -> ~320 cycles per K-block).
// Every mbarrier wait is bounded (mbar_wait); on expiry the kernel records a
// timeout in the status word and unwinds.
constexpr int kMxBM = 128;
constexpr int kMxBN = 256;
constexpr int kMxBK = 128;
constexpr int kMxStages = 4;
constexpr int kMxThreads = 320;
constexpr uint32_t kMxABytes = kMxBM * kMxBK;  // 16 KB
constexpr uint32_t kMxBBytes = kMxBN * kMxBK;  // 32 KB
constexpr uint32_t kMxSfBytes = 512 + 1024;    // A chunk + two B chunks
constexpr uint32_t kMxChunk = 32 * 32;         // epilogue staging chunk: 32 rows x 32 bytes
constexpr uint32_t kMxOffA = 0;
constexpr uint32_t kMxOffB = kMxOffA + kMxStages * kMxABytes;
constexpr uint32_t kMxOffSf = kMxOffB + kMxStages * kMxBBytes;
constexpr uint32_t kMxOffStage = kMxOffSf + kMxStages * kMxSfBytes;
constexpr uint32_t kMxOffBar = kMxOffStage + 8 * 2 * kMxChunk;
constexpr uint32_t kMxOffMisc = kMxOffBar + 16 * 8;
constexpr uint32_t kMxSmem = kMxOffMisc + 16 + 1024;  // + alignment slack
constexpr uint32_t kMxTmemCols = 512;
constexpr uint32_t kMxSfCol0 = 256;

struct MxGemmArgs {
  const uint8_t* sA;  // [K/128][tiles_m][512]
  const uint8_t* sB;  // [K/128][N/128][512]
  int64_t M;
  int64_t N;
  int64_t K;
  int tiles_m;
  int tiles_n;
};

template <bool kOutF32>
__global__ void __launch_bounds__(kMxThreads, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const MxGemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + kMxOffBar;           // [kMxStages]
  const uint32_t bar_empty = bar_full + kMxStages * 8;   // [kMxStages]
  const uint32_t bar_tfull = bar_empty + kMxStages * 8;  // accumulator complete
  const uint32_t bar_tempty = bar_tfull + 8;             // accumulator drained
  const uint32_t bar_drain = bar_tempty + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMxOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMxOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t KB = args.K / kMxBK;
  const int num_tiles = args.tiles_m * args.tiles_n;
  const int64_t rt_b = args.N / 128;  // B row tiles (scale chunks per K-block)

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMxStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_tfull, 1);
    mbar_init(bar_tempty, 8);  // one arrive per epilogue warp
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kMxTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // the whole warp runs the loop; one elected lane issues the copies
    uint32_t stage = 0, phase = 0, issued = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
      const int mt = t % args.tiles_m;
      const int nt = t / args.tiles_m;
      const bool full_n = static_cast<int64_t>(nt) * kMxBN + kMxBN <= args.N;
      for (int64_t kb = 0; kb < KB; ++kb) {
        if (!mbar_wait_warp(bar_empty + 8 * stage, phase ^ 1u, abort_flag)) { ok = false; break; }
        if (elect_one()) {
          const uint32_t sf = sbase + kMxOffSf + stage * kMxSfBytes;
          mbar_arrive_expect_tx(bar_full + 8 * stage, kMxABytes + kMxBBytes + kMxSfBytes);
          tma_load_2d(sbase + kMxOffA + stage * kMxABytes, &tmA, static_cast<int32_t>(kb * kMxBK), mt * kMxBM,
                      bar_full + 8 * stage);
          tma_load_2d(sbase + kMxOffB + stage * kMxBBytes, &tmB, static_cast<int32_t>(kb * kMxBK), nt * kMxBN,
                      bar_full + 8 * stage);
          bulk_load(sf, args.sA + (kb * args.tiles_m + mt) * 512, 512u, bar_full + 8 * stage);
          const uint8_t* sb = args.sB + (kb * rt_b + 2 * static_cast<int64_t>(nt)) * 512;
          if (full_n) {
            bulk_load(sf + 512, sb, 1024u, bar_full + 8 * stage);
          } else {
            // a 128-column tail tile: its rows 128-255 are zero-filled by
            // TMA, so any finite scale serves; repeat the first chunk
            bulk_load(sf + 512, sb, 512u, bar_full + 8 * stage);
            bulk_load(sf + 1024, sb, 512u, bar_full + 8 * stage);
          }
        }
        __syncwarp();
        ++issued;
        if (++stage == kMxStages) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok && lane == 0) {
      // drain: wait (bounded) for the copies still in flight
      for (uint32_t i = 0; i < kMxStages && i < issued; ++i) {
        if (stage == 0) { stage = kMxStages; phase ^= 1u; }
        --stage;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar_full + 8 * stage, phase) && globaltimer_ns() - t0 < 1000000ull) {}
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // the whole warp runs the loop (operands stay warp-uniform); one elected
    // lane issues the scale copies, the MMAs and the commits
    uint32_t stage = 0, phase = 0, tphase = 0;
    bool ok = true, any = false;
    for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
      // the previous tile's accumulator has been read out
      if (!mbar_wait_warp(bar_tempty, tphase ^ 1u, abort_flag)) { ok = false; break; }
      for (int64_t kb = 0; kb < KB; ++kb) {
        if (!mbar_wait_warp(bar_full + 8 * stage, phase, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sf = sbase + kMxOffSf + stage * kMxSfBytes;
        const uint32_t sfa = tmem_base + kMxSfCol0 + 32u * stage;
        const uint32_t sfb = sfa + 16u;
        const uint64_t adesc = smem_desc_k_sw128(sbase + kMxOffA + stage * kMxABytes);
        const uint64_t bdesc = smem_desc_k_sw128(sbase + kMxOffB + stage * kMxBBytes);
        if (elect_one()) {
          tmem_cp_32x128b_warpx4(sfa, smem_desc_rows16(sf));
          tmem_cp_32x128b_warpx4(sfb, smem_desc_rows16(sf + 512));
          tmem_cp_32x128b_warpx4(sfb + 4u, smem_desc_rows16(sf + 1024));
#pragma unroll
          for (int k = 0; k < kMxBK / 32; ++k)
            mma_mxf8f6f4(tmem_base, adesc + 2u * k, bdesc + 2u * k, idesc_mx_e4m3(kMxBM, kMxBN, k), sfa, sfb,
                         (kb | k) != 0 ? 1u : 0u);
          mma_commit(bar_empty + 8 * stage);
        }
        __syncwarp();
        any = true;
        if (++stage == kMxStages) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (elect_one()) mma_commit(bar_tfull);
      __syncwarp();
      tphase ^= 1u;
    }
    if (!ok && any && elect_one()) {
      // drain: wait (bounded) until every MMA issued is done; the commit is
      // made by the elected lane, the one that issued them
      mma_commit(bar_drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bar_drain, 0) && globaltimer_ns() - t0 < 1000000ull) {}
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;         // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;  // column half of the tile
    const uint32_t t_lane = static_cast<uint32_t>(q * 32) << 16;
    uint32_t tphase = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      const int mt = t % args.tiles_m;
      const int nt = t / args.tiles_m;
      const int64_t nh = static_cast<int64_t>(nt) * kMxBN + h * 128;
      const int64_t wrow0 = static_cast<int64_t>(mt) * kMxBM + q * 32;
      if (!mbar_wait_warp(bar_tfull, tphase, abort_flag)) break;
      tphase ^= 1u;
      __syncwarp();
      tc_fence_after();
      uint32_t p0[64], p1[64];
      tmem_ld_32x32b_x64(tmem_base + t_lane + h * 128, p0);
      tmem_ld_32x32b_x64(tmem_base + t_lane + h * 128 + 64, p1);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty);  // the next tile's MMAs may overwrite it
      if (nh >= args.N || wrow0 >= args.M) continue;
      // 32 rows x 128 columns out through shared memory and TMA stores in
      // 32-row x 32-byte chunks; TMA clips rows past the end of C
      uint8_t* stg = smem + kMxOffStage + (warp - 2) * 2 * kMxChunk;
      constexpr int kCols = kOutF32 ? 8 : 16;  // columns per 32-byte chunk row
#pragma unroll
      for (int c = 0; c < 128 / kCols; ++c) {
        uint8_t* cb = stg + (c & 1) * kMxChunk;
        if (lane == 0) bulk_wait_read<1>();  // the chunk buffer's previous store has read it
        __syncwarp();
        const uint32_t* src = (c * kCols < 64) ? p0 + c * kCols : p1 + (c * kCols - 64);
        uint4 v0, v1;
        if constexpr (kOutF32) {
          v0 = make_uint4(src[0], src[1], src[2], src[3]);
          v1 = make_uint4(src[4], src[5], src[6], src[7]);
        } else {
          v0 = make_uint4(cvt_bf16x2(__uint_as_float(src[0]), __uint_as_float(src[1])),
                          cvt_bf16x2(__uint_as_float(src[2]), __uint_as_float(src[3])),
                          cvt_bf16x2(__uint_as_float(src[4]), __uint_as_float(src[5])),
                          cvt_bf16x2(__uint_as_float(src[6]), __uint_as_float(src[7])));
          v1 = make_uint4(cvt_bf16x2(__uint_as_float(src[8]), __uint_as_float(src[9])),
                          cvt_bf16x2(__uint_as_float(src[10]), __uint_as_float(src[11])),
                          cvt_bf16x2(__uint_as_float(src[12]), __uint_as_float(src[13])),
                          cvt_bf16x2(__uint_as_float(src[14]), __uint_as_float(src[15])));
        }
        *reinterpret_cast<uint4*>(cb + lane * 32) = v0;
        *reinterpret_cast<uint4*>(cb + lane * 32 + 16) = v1;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmC, smem_u32(cb), static_cast<int32_t>(nh + c * kCols), static_cast<int32_t>(wrow0));
          bulk_commit();
        }
      }
    }
    // every TMA store of this warp has completed before the CTA exits
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kMxTmemCols);
  }
}

}  // namespace fp8q
