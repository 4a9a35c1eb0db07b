// fp8q.cu -- libfp8q.so: the C ABI declared in include/fp8q.h.
//
// Host side only validates arguments, builds TMA tensor maps and launches
// the kernels of quantize.cuh / gemm.cuh / mx.cuh on the caller's stream.  It never
// allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>

#include "fp8q.h"
#include "diag.cuh"
#include "gemm.cuh"
#include "mx.cuh"
#include "quantize.cuh"

namespace {

using namespace fp8q;

constexpr int kVersion = 100;  // 0.1.0

struct DeviceInfo {
  bool ok = false;
  int sms = 0;
};

// Per-device facts, probed once per device.
DeviceInfo device_info(int dev) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  static bool probed[64] = {};
  if (dev < 0 || dev >= 64) return DeviceInfo{};
  std::lock_guard<std::mutex> lock(mu);
  if (!probed[dev]) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) {
      cache[dev].ok = (major == 10 && minor == 3);
      cache[dev].sms = sms;
    }
    probed[dev] = true;
  }
  return cache[dev];
}

int check_device(DeviceInfo* out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FP8Q_ERR_CUDA;
  DeviceInfo di = device_info(dev);
  if (!di.ok) return FP8Q_ERR_DEVICE;
  if (out) *out = di;
  return FP8Q_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// cuTensorMapEncodeTiled through the runtime's driver entry point (no
// link-time dependency on libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D uint8 tensor [rows][cols] (cols contiguous), box 128 bytes x box_rows,
// 128-byte swizzle.  Out-of-range elements of a box read as zero.
bool make_tmap_u8(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {128u, box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D BF16 input [rows][cols] (cols contiguous), box 128 columns (256 bytes)
// x 128 rows, dense (no swizzle).  Out-of-range elements read as zero.
bool make_tmap_bf16_tile(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {128u, 128u};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D output tensor C [rows][cols] (BF16 or FP32, cols contiguous) for TMA
// stores of 32-row x 32-byte boxes, no swizzle.
bool make_tmap_out(CUtensorMap* tm, void* base, bool f32, uint64_t cols, uint64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const uint32_t esize = f32 ? 4u : 2u;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * esize};
  cuuint32_t box[2] = {32u / esize, 32u};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(tm, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int launch_status() { return cudaGetLastError() == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA; }

template <bool kF32, int kMode>
int launch_quant(const QuantArgs& a, int64_t grid_x, int64_t grid_y, cudaStream_t stream) {
  if (grid_y > 65535) return FP8Q_ERR_SHAPE;
  quant_tile_kernel<kF32, kMode><<<dim3(static_cast<unsigned>(grid_x), static_cast<unsigned>(grid_y)), 128, 0,
                                   stream>>>(a);
  return launch_status();
}

// BF16 input: the persistent double-buffered kernel, as many CTAs as fit on
// the device at once (occupancy probed once per device).
template <int kMode>
int launch_quant_pipe(const QuantArgs& a, int64_t tiles, cudaStream_t stream) {
  static std::atomic<int> resident[64];
  DeviceInfo di;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8Q_ERR_CUDA;
  const int st = check_device(&di);
  if (st != FP8Q_OK) return st;
  auto kern = quant_pipe_kernel<kMode>;
  constexpr int kSmem = 2 * kPipeTileBytes;
  int per_sm = resident[dev].load(std::memory_order_relaxed);
  if (per_sm == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 128, kSmem) != cudaSuccess)
      return FP8Q_ERR_CUDA;
    if (per_sm < 1) per_sm = 1;
    resident[dev].store(per_sm, std::memory_order_relaxed);
  }
  const int64_t cap = static_cast<int64_t>(di.sms) * per_sm;
  const int grid = static_cast<int>(tiles < cap ? tiles : cap);
  kern<<<grid, 128, kSmem, stream>>>(a, tiles);
  return launch_status();
}

// BF16 through the split-role persistent kernel (one 128-thread warpgroup
// per output), as many CTAs as fit on the device (occupancy probed once per
// device).
template <bool kRow, bool kCol, bool kBlk, bool kMx = false>
int launch_quant_rc(const QuantArgs& a, int64_t tiles, cudaStream_t stream) {
  static std::atomic<int> resident[64];
  DeviceInfo di;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8Q_ERR_CUDA;
  const int st = check_device(&di);
  if (st != FP8Q_OK) return st;
  auto kern = quant_rc_kernel<kRow, kCol, kBlk, kMx>;
  constexpr int kSmem = rc_smem_bytes(kRow, kCol);
  constexpr int kThreads = (kRow ? 128 : 0) + (kCol ? 128 : 0);
  int per_sm = resident[dev].load(std::memory_order_relaxed);
  if (per_sm == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, kSmem) != cudaSuccess)
      return FP8Q_ERR_CUDA;
    if (per_sm < 1) per_sm = 1;
    resident[dev].store(per_sm, std::memory_order_relaxed);
  }
  // the code tiles leave through TMA stores (128-byte swizzle, 128 x 128 boxes)
  CUtensorMap tm_x, tm_row, tm_col;
  std::memset(&tm_row, 0, sizeof(tm_row));
  std::memset(&tm_col, 0, sizeof(tm_col));
  if (!make_tmap_bf16_tile(&tm_x, a.x, static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.M)))
    return FP8Q_ERR_CUDA;
  if (kRow && !make_tmap_u8(&tm_row, kBlk ? a.q_blk : a.q_row, static_cast<uint64_t>(a.K),
                            static_cast<uint64_t>(a.M), 128))
    return FP8Q_ERR_CUDA;
  if (kCol && !make_tmap_u8(&tm_col, kBlk ? a.q_blkT : a.q_colT, static_cast<uint64_t>(a.M),
                            static_cast<uint64_t>(a.K), 128))
    return FP8Q_ERR_CUDA;
  const int64_t cap = static_cast<int64_t>(di.sms) * per_sm;
  const int grid = static_cast<int>(tiles < cap ? tiles : cap);
  kern<<<grid, kThreads, kSmem, stream>>>(a, tiles, tm_x, tm_row, tm_col);
  return launch_status();
}

// FP32 input: one CTA per tile.  BF16: the TMA-fed split-role kernel, one
// warpgroup per output (rows, transposed columns, blocks with their
// transpose, or either alone), except for the row gather (scattered rows:
// the pipelined kernel's one bulk copy per row) and 128x128 blocks without
// the transpose, where the pipelined kernel's 12 warps per SM measured
// faster than one warpgroup per CTA (5.72 vs 5.48 TB/s on 18432 x 7168).
template <int kMode>
int launch_quant_dt(int in_dtype, const QuantArgs& a, int64_t gx, int64_t gy, cudaStream_t s) {
  if (in_dtype == FP8Q_FP32) return launch_quant<true, kMode>(a, gx, gy, s);
  if constexpr (kMode == (kQRow | kQCol)) return launch_quant_rc<true, true, false>(a, gx * gy, s);
  if constexpr (kMode == kQCol) return launch_quant_rc<false, true, false>(a, gx * gy, s);
  if constexpr (kMode == (kQBlk | kQBlkT)) return launch_quant_rc<true, true, true>(a, gx * gy, s);
  if constexpr (kMode == kQBlkT) return launch_quant_rc<false, true, true>(a, gx * gy, s);
  if constexpr (kMode == kQRow) {
    if (a.src_rows == nullptr) return launch_quant_rc<true, false, false>(a, gx * gy, s);
  }
  return launch_quant_pipe<kMode>(a, gx * gy, s);
}

// One CTA per SM (persistent).  A stream-K launch is cooperative: its CTAs
// wait on each other's partial tiles, so they must all be resident at once.
template <bool kOutF32, int kSbGran, bool kGrouped, bool kStreamK, bool kRing>
int launch_gemm_k(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const GemmArgs& a, int grid,
                  cudaStream_t s) {
  auto kern = gemm_kernel<kOutF32, kSbGran, kGrouped, kStreamK, kRing>;
  const uint32_t smem = gemm_smem_bytes(kSbGran, kGrouped);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return FP8Q_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = a.streamk ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, a) != cudaSuccess) return FP8Q_ERR_CUDA;
  return launch_status();
}

// Scales go through the shared-memory ring for per-column B scales, the
// grouped form, stream-K and long K (more than 64 K-blocks: 2187 against 1907
// TFLOP/s at K = 18432); a dense short-K data-parallel GEMM loads them in the
// promotion warps (2468 against 2357 TFLOP/s at K = 7168).
template <bool kOutF32, int kSbGran, bool kGrouped>
int launch_gemm_t(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const GemmArgs& a, int grid,
                  cudaStream_t s) {
  if constexpr (kGrouped || kSbGran == 1) {
    return a.streamk ? launch_gemm_k<kOutF32, kSbGran, kGrouped, !kGrouped, true>(ta, tb, tc, a, grid, s)
                     : launch_gemm_k<kOutF32, kSbGran, kGrouped, false, true>(ta, tb, tc, a, grid, s);
  } else {
    const bool ring = a.K / kBK > 64;
    // stream-K always takes the scale ring: the variant with per-thread
    // scale loads spills there (4096x7168x7168: 17% slower)
    if (a.streamk) return launch_gemm_k<kOutF32, kSbGran, false, true, true>(ta, tb, tc, a, grid, s);
    return ring ? launch_gemm_k<kOutF32, kSbGran, false, false, true>(ta, tb, tc, a, grid, s)
                : launch_gemm_k<kOutF32, kSbGran, false, false, false>(ta, tb, tc, a, grid, s);
  }
}

// Stream-K workspace: [flags: one u32 per CTA, padded to 256 bytes]
// [partial tiles: one 128 x 256 FP32 tile per CTA].
constexpr size_t kPartialBytes = static_cast<size_t>(kBM) * kBN * 4;
size_t workspace_bytes_for(int ctas) {
  return ((static_cast<size_t>(ctas) * 4 + 255) & ~size_t(255)) + static_cast<size_t>(ctas) * kPartialBytes;
}

// Call epochs for the stream-K flags: never 0 (the idle value).
uint32_t next_epoch() {
  static std::atomic<uint32_t> counter{0};
  uint32_t e = counter.fetch_add(1, std::memory_order_relaxed) + 1;
  if (e == 0) e = counter.fetch_add(1, std::memory_order_relaxed) + 1;
  return e;
}

int gemm_common(const uint8_t* Aq, const float* sA, const uint8_t* Bq, const float* sB, void* C, int64_t M,
                int64_t N, int64_t K, int out_dtype, int sb_gran, const int32_t* row_offsets, int32_t E,
                cudaStream_t stream, void* workspace = nullptr, size_t workspace_bytes = 0) {
  const bool grouped = row_offsets != nullptr;
  if (out_dtype != FP8Q_BF16 && out_dtype != FP8Q_FP32) return FP8Q_ERR_DTYPE;
  if (sb_gran != 128 && sb_gran != 1) return FP8Q_ERR_DTYPE;
  if (M < 0 || N <= 0 || K <= 0 || N % 128 != 0 || K % 128 != 0) return FP8Q_ERR_SHAPE;
  if (grouped && (E < 1 || E > kMaxExperts)) return FP8Q_ERR_SHAPE;
  if (M > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 31) - 1)
    return FP8Q_ERR_SHAPE;
  if (grouped && static_cast<int64_t>(E) * N > (int64_t(1) << 31) - 1) return FP8Q_ERR_SHAPE;
  if (M == 0) return FP8Q_OK;  // empty operands may carry null pointers
  if (!Aq || !sA || !Bq || !sB || !C) return FP8Q_ERR_NULL;
  if (!aligned16(Aq) || !aligned16(sA) || !aligned16(Bq) || !aligned16(sB) || !aligned16(C) ||
      (grouped && !aligned16(row_offsets)) || (workspace && !aligned16(workspace)))
    return FP8Q_ERR_ALIGN;
  DeviceInfo di;
  int st = check_device(&di);
  if (st != FP8Q_OK) return st;

  CUtensorMap ta, tb;
  if (!make_tmap_u8(&ta, Aq, static_cast<uint64_t>(K), static_cast<uint64_t>(M), kBM)) return FP8Q_ERR_CUDA;
  const uint64_t brows = grouped ? static_cast<uint64_t>(E) * N : static_cast<uint64_t>(N);
  if (!make_tmap_u8(&tb, Bq, static_cast<uint64_t>(K), brows, kBN)) return FP8Q_ERR_CUDA;
  CUtensorMap tc;
  if (!make_tmap_out(&tc, C, out_dtype == FP8Q_FP32, static_cast<uint64_t>(N), static_cast<uint64_t>(M)))
    return FP8Q_ERR_CUDA;

  GemmArgs a;
  a.sA = sA;
  a.lds_a = M;
  a.sB = sB;
  a.C = C;
  a.M = M;
  a.N = N;
  a.K = K;
  a.tiles_m = static_cast<int>((M + kBM - 1) / kBM);
  a.tiles_n = static_cast<int>((N + kBN - 1) / kBN);
  // Raster order.  Concurrent CTAs walk K in step, so a wave reads the A rows
  // of all its M-tiles once; when A is too large to stay in L2 from one wave
  // to the next (K = 18432 Dgrad: 75 MB of codes, re-read by each of 6 waves)
  // tiles go in groups of 16 M-tiles over all N-tiles, which halves the A
  // rows a wave touches (measured 1.6% faster there, same elsewhere).
  constexpr int kMGroup = 16;
  a.m_group = (M * K > (int64_t(64) << 20) && a.tiles_m > kMGroup) ? kMGroup : a.tiles_m;
  a.row_offsets = row_offsets;
  a.E = grouped ? E : 1;
  a.streamk = 0;
  a.sk_tile0 = 0;
  a.sa_bulk = (M % 4 == 0) ? 1 : 0;  // lds_a == M; sA itself is 16-byte aligned (checked above)
  a.ws = nullptr;
  a.flags = nullptr;
  a.epoch = 0;

  int64_t tiles_upper;
  if (grouped) {
    tiles_upper = (static_cast<int64_t>(a.tiles_m) + E) * a.tiles_n;
  } else {
    tiles_upper = static_cast<int64_t>(a.tiles_m) * a.tiles_n;
  }
  if (tiles_upper > (int64_t(1) << 31) - 1) return FP8Q_ERR_SHAPE;
  int grid = static_cast<int>(tiles_upper < di.sms ? tiles_upper : di.sms);
  if (workspace != nullptr && !grouped) {
    if (workspace_bytes < workspace_bytes_for(di.sms)) return FP8Q_ERR_WORKSPACE;
    // stream-K when whole tiles leave the last wave of the persistent grid
    // less than 95% busy (or there are fewer tiles than SMs)
    const int64_t waves = (tiles_upper + di.sms - 1) / di.sms;
    const int64_t kb_total = tiles_upper * (K / kBK);
    if (tiles_upper * 100 < waves * di.sms * 95 && kb_total >= di.sms &&
        kb_total < (int64_t(1) << 62) / di.sms) {
      grid = di.sms;
      a.streamk = 1;
      // whole-tile waves first, the last full wave plus the remainder
      // balanced by stream-K
      a.sk_tile0 = static_cast<int>(waves >= 2 ? (waves - 2) * di.sms : 0);
      a.flags = static_cast<uint32_t*>(workspace);
      a.ws = reinterpret_cast<float4*>(static_cast<uint8_t*>(workspace) +
                                       ((static_cast<size_t>(di.sms) * 4 + 255) & ~size_t(255)));
      a.epoch = next_epoch();
    }
  }
  const bool f32 = out_dtype == FP8Q_FP32;
  if (grouped) {
    return f32 ? launch_gemm_t<true, 128, true>(ta, tb, tc, a, grid, stream)
               : launch_gemm_t<false, 128, true>(ta, tb, tc, a, grid, stream);
  }
  if (sb_gran == 1) {
    return f32 ? launch_gemm_t<true, 1, false>(ta, tb, tc, a, grid, stream)
               : launch_gemm_t<false, 1, false>(ta, tb, tc, a, grid, stream);
  }
  return f32 ? launch_gemm_t<true, 128, false>(ta, tb, tc, a, grid, stream)
             : launch_gemm_t<false, 128, false>(ta, tb, tc, a, grid, stream);
}

// MX variant: bytes of the tiled E8M0 scale array of a rows x K operand.
size_t mx_scale_bytes(int64_t rows, int64_t K) {
  return static_cast<size_t>(K / 128) * static_cast<size_t>((rows + 127) / 128) * 512u;
}

template <bool kF32>
int launch_quant_mx(const void* x, int64_t rows, int64_t K, uint8_t* q, uint8_t* s, cudaStream_t stream) {
  static std::atomic<int> resident[64];
  DeviceInfo di;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8Q_ERR_CUDA;
  const int st = check_device(&di);
  if (st != FP8Q_OK) return st;
  auto kern = quant_mx_kernel<kF32>;
  int per_sm = resident[dev].load(std::memory_order_relaxed);
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kMxQuantThreads, 0) != cudaSuccess)
      return FP8Q_ERR_CUDA;
    if (per_sm < 1) per_sm = 1;
    resident[dev].store(per_sm, std::memory_order_relaxed);
  }
  const int64_t slabs = (K / 128) * ((rows + 127) / 128) * 8;  // 16-row x 128-column slabs, one per warp
  const int64_t cap = static_cast<int64_t>(di.sms) * per_sm;
  const int64_t need = (slabs + kMxQuantThreads / 32 - 1) / (kMxQuantThreads / 32);
  const int grid = static_cast<int>(need < cap ? need : cap);
  kern<<<grid, kMxQuantThreads, 0, stream>>>(x, rows, K, q, s, slabs);
  return launch_status();
}

int mx_gemm_common(const uint8_t* Aq, const uint8_t* sA, const uint8_t* Bq, const uint8_t* sB, void* C, int64_t M,
                   int64_t N, int64_t K, int out_dtype, cudaStream_t stream) {
  if (out_dtype != FP8Q_BF16 && out_dtype != FP8Q_FP32) return FP8Q_ERR_DTYPE;
  if (M < 0 || N <= 0 || K <= 0 || N % 128 != 0 || K % 128 != 0) return FP8Q_ERR_SHAPE;
  if (M > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 31) - 1)
    return FP8Q_ERR_SHAPE;
  const int64_t tiles_m = (M + kMxBM - 1) / kMxBM, tiles_n = (N + kMxBN - 1) / kMxBN;
  if (tiles_m * tiles_n > (int64_t(1) << 31) - 1) return FP8Q_ERR_SHAPE;
  if (M == 0) return FP8Q_OK;  // empty operands may carry null pointers
  if (!Aq || !sA || !Bq || !sB || !C) return FP8Q_ERR_NULL;
  if (!aligned16(Aq) || !aligned16(sA) || !aligned16(Bq) || !aligned16(sB) || !aligned16(C)) return FP8Q_ERR_ALIGN;
  DeviceInfo di;
  const int st = check_device(&di);
  if (st != FP8Q_OK) return st;
  CUtensorMap ta, tb, tc;
  if (!make_tmap_u8(&ta, Aq, static_cast<uint64_t>(K), static_cast<uint64_t>(M), kMxBM)) return FP8Q_ERR_CUDA;
  if (!make_tmap_u8(&tb, Bq, static_cast<uint64_t>(K), static_cast<uint64_t>(N), kMxBN)) return FP8Q_ERR_CUDA;
  if (!make_tmap_out(&tc, C, out_dtype == FP8Q_FP32, static_cast<uint64_t>(N), static_cast<uint64_t>(M)))
    return FP8Q_ERR_CUDA;
  MxGemmArgs a;
  a.sA = sA;
  a.sB = sB;
  a.M = M;
  a.N = N;
  a.K = K;
  a.tiles_m = static_cast<int>(tiles_m);
  a.tiles_n = static_cast<int>(tiles_n);
  const int64_t tiles = tiles_m * tiles_n;
  const int grid = static_cast<int>(tiles < di.sms ? tiles : di.sms);
  auto kern = out_dtype == FP8Q_FP32 ? gemm_mx_kernel<true> : gemm_mx_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kMxSmem)) !=
      cudaSuccess)
    return FP8Q_ERR_CUDA;
  kern<<<grid, kMxThreads, kMxSmem, stream>>>(ta, tb, tc, a);
  return launch_status();
}

}  // namespace

// ---------------------------------------------------------------------------
// Library-owned stream-K scratch for fp8q_gemm_ws_static.  For callers that
// have no allocator at hand -- e.g. a plugin or operator interface whose
// enqueue step is handed only its input and output buffers, or a path that
// must not take cudaMalloc's implicit device-wide synchronization -- the
// workspace fp8q_gemm_ws would need lives in this fixed array instead.  It is
// sized for a grid of up to kStaticScratchCtas CTAs (one per SM), about
// 20 MB, and every GPU that loads the library holds it until the process
// exits.
// ---------------------------------------------------------------------------
constexpr int kStaticScratchCtas = 160;
constexpr size_t kStaticScratchBytes = ((static_cast<size_t>(kStaticScratchCtas) * 4 + 255) & ~size_t(255)) +
                                       static_cast<size_t>(kStaticScratchCtas) * (static_cast<size_t>(kBM) * kBN * 4);
static __device__ __align__(256) unsigned char g_gemm_scratch[kStaticScratchBytes];

namespace {

// Device address of g_gemm_scratch on the current device.  In host code the
// array's name is only a host-side handle, so the address is looked up once
// per device (with that device current) and cached.
int static_scratch(void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8Q_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_gemm_scratch) != cudaSuccess || p == nullptr) return FP8Q_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return FP8Q_OK;
}

}  // namespace

extern "C" {

int fp8q_version(void) { return kVersion; }

const char* fp8q_status_string(int status) {
  switch (status) {
    case FP8Q_OK: return "ok";
    case FP8Q_ERR_NULL: return "null pointer argument";
    case FP8Q_ERR_SHAPE: return "invalid shape (negative size or divisibility rule broken)";
    case FP8Q_ERR_ALIGN: return "pointer not 16-byte aligned";
    case FP8Q_ERR_DTYPE: return "unknown dtype or granularity code";
    case FP8Q_ERR_DEVICE: return "current device is not sm_103 (B300)";
    case FP8Q_ERR_CUDA: return "CUDA call or kernel launch failed";
    case FP8Q_ERR_TIMEOUT: return "a kernel pipeline wait timed out on the device";
    case FP8Q_ERR_WORKSPACE: return "workspace smaller than fp8q_gemm_workspace_size()";
    default: return "unknown status";
  }
}

int fp8q_quantize_act(const void* x, int in_dtype, int64_t M, int64_t K, uint8_t* q_row, float* s_row,
                      uint8_t* q_colT, float* s_col, fp8q_stream_t stream) {
  const bool row = q_row != nullptr || s_row != nullptr;
  const bool col = q_colT != nullptr || s_col != nullptr;
  if (in_dtype != FP8Q_BF16 && in_dtype != FP8Q_FP32) return FP8Q_ERR_DTYPE;
  if (M < 0 || K <= 0 || K % 128 != 0) return FP8Q_ERR_SHAPE;
  if (col && M % 128 != 0) return FP8Q_ERR_SHAPE;
  if (M == 0) return FP8Q_OK;  // empty operands may carry null pointers
  if (!x) return FP8Q_ERR_NULL;
  if (!row && !col) return FP8Q_ERR_NULL;
  if ((row && (!q_row || !s_row)) || (col && (!q_colT || !s_col))) return FP8Q_ERR_NULL;
  if (!aligned16(x) || (row && (!aligned16(q_row) || !aligned16(s_row))) ||
      (col && (!aligned16(q_colT) || !aligned16(s_col))))
    return FP8Q_ERR_ALIGN;
  int st = check_device(nullptr);
  if (st != FP8Q_OK) return st;
  QuantArgs a{};
  a.x = x;
  a.M = M;
  a.K = K;
  a.q_row = q_row;
  a.s_row = s_row;
  a.ld_srow = M;
  a.q_colT = q_colT;
  a.s_col = s_col;
  const int64_t gx = K / 128, gy = (M + 127) / 128;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (row && col) return launch_quant_dt<kQRow | kQCol>(in_dtype, a, gx, gy, s);
  if (row) return launch_quant_dt<kQRow>(in_dtype, a, gx, gy, s);
  return launch_quant_dt<kQCol>(in_dtype, a, gx, gy, s);
}

int fp8q_quantize_act_gather(const void* x, int in_dtype, int64_t M, int64_t K, const int32_t* src_rows, int64_t R,
                             uint8_t* q_row, float* s_row, fp8q_stream_t stream) {
  if (in_dtype != FP8Q_BF16 && in_dtype != FP8Q_FP32) return FP8Q_ERR_DTYPE;
  if (M < 0 || R < 0 || K <= 0 || K % 128 != 0) return FP8Q_ERR_SHAPE;
  if (R > 0 && M == 0) return FP8Q_ERR_SHAPE;
  if (R == 0) return FP8Q_OK;  // empty operands may carry null pointers
  if (!x || !src_rows || !q_row || !s_row) return FP8Q_ERR_NULL;
  if (!aligned16(x) || !aligned16(src_rows) || !aligned16(q_row) || !aligned16(s_row)) return FP8Q_ERR_ALIGN;
  int st = check_device(nullptr);
  if (st != FP8Q_OK) return st;
  QuantArgs a{};
  a.x = x;
  a.M = R;
  a.K = K;
  a.src_rows = src_rows;
  a.q_row = q_row;
  a.s_row = s_row;
  a.ld_srow = R;
  return launch_quant_dt<kQRow>(in_dtype, a, K / 128, (R + 127) / 128, reinterpret_cast<cudaStream_t>(stream));
}

int fp8q_quantize_weight_ex(const void* w, int in_dtype, int64_t N, int64_t K, uint8_t* q, float* s, uint8_t* q_t,
                            float* s_t, fp8q_stream_t stream) {
  const bool fw = q != nullptr || s != nullptr;
  const bool tr = q_t != nullptr || s_t != nullptr;
  if (in_dtype != FP8Q_BF16 && in_dtype != FP8Q_FP32) return FP8Q_ERR_DTYPE;
  if (N < 0 || K <= 0 || N % 128 != 0 || K % 128 != 0) return FP8Q_ERR_SHAPE;
  if (N == 0) return FP8Q_OK;  // empty operands may carry null pointers
  if (!w) return FP8Q_ERR_NULL;
  if (!fw && !tr) return FP8Q_ERR_NULL;
  if ((fw && (!q || !s)) || (tr && (!q_t || !s_t))) return FP8Q_ERR_NULL;
  if (!aligned16(w) || (fw && (!aligned16(q) || !aligned16(s))) || (tr && (!aligned16(q_t) || !aligned16(s_t))))
    return FP8Q_ERR_ALIGN;
  int st = check_device(nullptr);
  if (st != FP8Q_OK) return st;
  QuantArgs a{};
  a.x = w;
  a.M = N;
  a.K = K;
  a.q_blk = q;
  a.s_blk = s;
  a.q_blkT = q_t;
  a.s_blkT = s_t;
  const int64_t gx = K / 128, gy = N / 128;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (fw && tr) return launch_quant_dt<kQBlk | kQBlkT>(in_dtype, a, gx, gy, cs);
  if (fw) return launch_quant_dt<kQBlk>(in_dtype, a, gx, gy, cs);
  return launch_quant_dt<kQBlkT>(in_dtype, a, gx, gy, cs);
}

int fp8q_quantize_weight(const void* w, int in_dtype, int64_t N, int64_t K, uint8_t* q, float* s,
                         fp8q_stream_t stream) {
  if (N != 0 && (!q || !s)) return FP8Q_ERR_NULL;
  return fp8q_quantize_weight_ex(w, in_dtype, N, K, q, s, nullptr, nullptr, stream);
}

int fp8q_gemm(const uint8_t* Aq, const float* sA, const uint8_t* Bq, const float* sB, void* C, int64_t M, int64_t N,
              int64_t K, int out_dtype, fp8q_stream_t stream) {
  return gemm_common(Aq, sA, Bq, sB, C, M, N, K, out_dtype, 128, nullptr, 0, reinterpret_cast<cudaStream_t>(stream));
}

int fp8q_gemm_ex(const uint8_t* Aq, const float* sA, const uint8_t* Bq, const float* sB, void* C, int64_t M,
                 int64_t N, int64_t K, int out_dtype, int sb_gran_n, fp8q_stream_t stream) {
  return gemm_common(Aq, sA, Bq, sB, C, M, N, K, out_dtype, sb_gran_n, nullptr, 0,
                     reinterpret_cast<cudaStream_t>(stream));
}

size_t fp8q_gemm_workspace_size(void) {
  DeviceInfo di;
  if (check_device(&di) != FP8Q_OK) return 0;
  return workspace_bytes_for(di.sms);
}

int fp8q_gemm_ws(const uint8_t* Aq, const float* sA, const uint8_t* Bq, const float* sB, void* C, int64_t M,
                 int64_t N, int64_t K, int out_dtype, int sb_gran_n, void* workspace, size_t workspace_bytes,
                 fp8q_stream_t stream) {
  return gemm_common(Aq, sA, Bq, sB, C, M, N, K, out_dtype, sb_gran_n, nullptr, 0,
                     reinterpret_cast<cudaStream_t>(stream), workspace, workspace_bytes);
}

int fp8q_gemm_ws_static(const uint8_t* Aq, const float* sA, const uint8_t* Bq, const float* sB, void* C,
                        int64_t M, int64_t N, int64_t K, int out_dtype, int sb_gran_n, fp8q_stream_t stream) {
  DeviceInfo di;
  const int st = check_device(&di);
  if (st != FP8Q_OK) return st;
  // the grid (one CTA per SM) must fit the fixed scratch
  if (workspace_bytes_for(di.sms) > kStaticScratchBytes) return FP8Q_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int sst = static_scratch(&scratch);
  if (sst != FP8Q_OK) return sst;
  // the flag words must start at zero; clear them on this stream (earlier
  // calls leave them zero unless one stopped on a timeout)
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, static_cast<size_t>(di.sms) * 4, cs) != cudaSuccess) return FP8Q_ERR_CUDA;
  return gemm_common(Aq, sA, Bq, sB, C, M, N, K, out_dtype, sb_gran_n, nullptr, 0, cs, scratch, kStaticScratchBytes);
}

int fp8q_gemm_unpromoted(const uint8_t* Aq, const uint8_t* Bq, float* C, int64_t M, int64_t N, int64_t K,
                         fp8q_stream_t stream) {
  if (M < 0 || N <= 0 || K <= 0 || N % 128 != 0 || K % 128 != 0) return FP8Q_ERR_SHAPE;
  if (M > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 31) - 1)
    return FP8Q_ERR_SHAPE;
  if (M == 0) return FP8Q_OK;
  if (!Aq || !Bq || !C) return FP8Q_ERR_NULL;
  if (!aligned16(Aq) || !aligned16(Bq) || !aligned16(C)) return FP8Q_ERR_ALIGN;
  const int st = check_device(nullptr);
  if (st != FP8Q_OK) return st;
  CUtensorMap ta, tb;
  if (!make_tmap_u8(&ta, Aq, static_cast<uint64_t>(K), static_cast<uint64_t>(M), kDiagBM)) return FP8Q_ERR_CUDA;
  if (!make_tmap_u8(&tb, Bq, static_cast<uint64_t>(K), static_cast<uint64_t>(N), kDiagBN)) return FP8Q_ERR_CUDA;
  if (cudaFuncSetAttribute(gemm_unpromoted_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kDiagSmem)) != cudaSuccess)
    return FP8Q_ERR_CUDA;
  const dim3 grid(static_cast<unsigned>((M + kDiagBM - 1) / kDiagBM), static_cast<unsigned>((N + kDiagBN - 1) / kDiagBN));
  if (grid.x > 2147483647u || grid.y > 65535u) return FP8Q_ERR_SHAPE;
  gemm_unpromoted_kernel<<<grid, 128, kDiagSmem, reinterpret_cast<cudaStream_t>(stream)>>>(ta, tb, C, M, N, K);
  return launch_status();
}

int fp8q_grouped_gemm(const uint8_t* Aq, const float* sA, const uint8_t* Bq, const float* sB, void* C,
                      const int32_t* row_offsets, int32_t E, int64_t total_rows, int64_t N, int64_t K, int out_dtype,
                      fp8q_stream_t stream) {
  if (!row_offsets && total_rows != 0) return FP8Q_ERR_NULL;
  if (!row_offsets) return E < 1 || E > kMaxExperts ? FP8Q_ERR_SHAPE : FP8Q_OK;
  return gemm_common(Aq, sA, Bq, sB, C, total_rows, N, K, out_dtype, 128, row_offsets, E,
                     reinterpret_cast<cudaStream_t>(stream));
}

size_t fp8q_mx_scale_bytes(int64_t rows, int64_t K) {
  if (rows < 0 || K <= 0 || K % 128 != 0) return 0;
  return mx_scale_bytes(rows, K);
}

int fp8q_mx_quantize(const void* x, int in_dtype, int64_t rows, int64_t K, uint8_t* q, uint8_t* s,
                     fp8q_stream_t stream) {
  if (in_dtype != FP8Q_BF16 && in_dtype != FP8Q_FP32) return FP8Q_ERR_DTYPE;
  if (rows < 0 || K <= 0 || K % 128 != 0) return FP8Q_ERR_SHAPE;
  if (rows == 0) return FP8Q_OK;  // empty operands may carry null pointers
  if (!x || !q || !s) return FP8Q_ERR_NULL;
  if (!aligned16(x) || !aligned16(q) || !aligned16(s)) return FP8Q_ERR_ALIGN;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (in_dtype == FP8Q_FP32) return launch_quant_mx<true>(x, rows, K, q, s, cs);
  // BF16: the TMA-fed split-role kernel's row path in MX mode
  const int st = check_device(nullptr);
  if (st != FP8Q_OK) return st;
  QuantArgs a{};
  a.x = x;
  a.M = rows;
  a.K = K;
  a.q_row = q;
  a.s_mx = s;
  return launch_quant_rc<true, false, false, true>(a, (K / 128) * ((rows + 127) / 128), cs);
}

int fp8q_mx_gemm(const uint8_t* Aq, const uint8_t* sA, const uint8_t* Bq, const uint8_t* sB, void* C, int64_t M,
                 int64_t N, int64_t K, int out_dtype, fp8q_stream_t stream) {
  return mx_gemm_common(Aq, sA, Bq, sB, C, M, N, K, out_dtype, reinterpret_cast<cudaStream_t>(stream));
}

int fp8q_selftest_wait_timeout(fp8q_stream_t stream) {
  const int st = check_device(nullptr);
  if (st != FP8Q_OK) return st;
  selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>();
  return launch_status();
}

int fp8q_get_device_status(fp8q_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FP8Q_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, fp8q::g_status_word, sizeof(v)) != cudaSuccess) return FP8Q_ERR_CUDA;
  if (v != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(fp8q::g_status_word, &zero, sizeof(zero)) != cudaSuccess) return FP8Q_ERR_CUDA;
  }
  return static_cast<int>(v);
}

}  // extern "C"
