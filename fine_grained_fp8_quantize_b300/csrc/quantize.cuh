// quantize.cuh -- HBM-bound fine-grained E4M3 quantizers for sm_103a.
//
// One CTA (4 warps, 128 threads) owns one 128 x 128 tile of the input.
// Thread (warp w, lane l) holds rows w*32 + (l/16)*16 + j (j = 0..15) and
// columns (l%16)*8 .. +7 of the tile in registers, loaded with 16-byte
// vector loads (a warp instruction reads two full 256-byte tile rows).
// From those registers it forms, as the mode asks:
//   ROW   1x128 groups (one row, 128 channels): activations
//         (dssusan.co.kr page, the Figure 7 (a) passage);
//   COL   128x1 groups (128 rows, one channel) stored transposed, the copy
//         FP8 Wgrad consumes ("Is aI Hitting a Wall?", the Wgrad sentence);
//   BLK   one 128x128 group: weights (same Figure 7 (a) passage), written
//         as-is and/or transposed (the Dgrad operand).
// Group scale: a = max(amax, 2^-100), s = a / 448, inv = 448 / a (IEEE
// single divisions, no fast-math), code = E4M3_rn_satfinite(x * inv).
// Row amax: warp shuffles over the 16 lanes sharing a row.  Column amax:
// shuffle across the two 16-row halves, then shared memory across warps.
// Codes leave as 8-byte row stores (a warp writes full 128-byte lines) and
// 16-byte transposed stores (a warp writes full 32-byte sectors).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "mx.cuh"
#include "ptx.cuh"

namespace fp8q {

enum QuantMode : int {
  kQRow = 1,    // 1x128 row groups   -> q_row[M][K], s_row[K/128][ld_srow]
  kQCol = 2,    // 128x1 column groups -> q_colT[K][M], s_col[M/128][K]
  kQBlk = 4,    // 128x128 block       -> q_blk[M][K], s_blk[M/128][K/128]
  kQBlkT = 8,   // 128x128 block, transposed codes -> q_blkT[K][M], s_blkT[K/128][M/128]
};

struct QuantArgs {
  const void* x;            // [rows_in][K] BF16 or FP32
  int64_t M;                // rows of the (gathered) problem
  int64_t K;                // columns, multiple of 128
  const int32_t* src_rows;  // row gather (ROW mode only) or nullptr
  uint8_t* q_row;
  float* s_row;
  int64_t ld_srow;          // row stride of s_row (= M)
  uint8_t* q_colT;
  float* s_col;
  uint8_t* q_blk;
  float* s_blk;
  uint8_t* q_blkT;
  float* s_blkT;
  uint8_t* s_mx;            // MX row mode: E8M0 scales in the tensor core's tiled layout
};

// 16 rows x 8 columns of the input held by one thread.
template <bool kF32>
struct Frag;

template <>
struct Frag<false> {  // BF16: 8 values per 16-byte word, kept packed
  uint4 v[16];
  __device__ __forceinline__ void load(const void* base, int64_t elem_off, int j) {
    v[j] = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + elem_off));
  }
  __device__ __forceinline__ void zero(int j) { v[j] = make_uint4(0u, 0u, 0u, 0u); }
  __device__ __forceinline__ float get(int j, int i) const {
    const uint32_t w = (i < 2) ? v[j].x : (i < 4) ? v[j].y : (i < 6) ? v[j].z : v[j].w;
    return (i & 1) ? bf16hi_to_f32(w) : bf16lo_to_f32(w);
  }
};

template <>
struct Frag<true> {  // FP32: 8 values in two 16-byte words
  float4 v[16][2];
  __device__ __forceinline__ void load(const void* base, int64_t elem_off, int j) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem_off);
    v[j][0] = __ldg(p);
    v[j][1] = __ldg(p + 1);
  }
  __device__ __forceinline__ void zero(int j) {
    v[j][0] = make_float4(0.f, 0.f, 0.f, 0.f);
    v[j][1] = v[j][0];
  }
  __device__ __forceinline__ float get(int j, int i) const {
    const float4& h = v[j][i >> 2];
    const int r = i & 3;
    return r == 0 ? h.x : r == 1 ? h.y : r == 2 ? h.z : h.w;
  }
};

// amax -> (s, inv).  IEEE round-to-nearest-even divisions (the build uses
// -prec-div=true and no fast-math, so '/' is div.rn.f32).
__device__ __forceinline__ void group_scale(float amax, float& s, float& inv) {
  const float a = fmaxf(amax, 0x1p-100f);
  s = __fdiv_rn(a, 448.0f);
  inv = __fdiv_rn(448.0f, a);
}

// Shared-memory scratch of one tile's column / block reductions.
struct QuantRed {
  float red[4][128];  // per-warp column maxima
  float inv[128];     // per-column inverse scales
  float blk[4];       // per-warp block maxima
};

// Everything after the load: group amax, scales, E4M3 casts and stores of
// the 128 x 128 tile (kb, mb) whose fragment this thread holds in `f`.
// Called by all 128 threads of the CTA (it synchronizes the CTA).
template <bool kF32, int kMode>
__device__ __forceinline__ void quant_tile_body(const Frag<kF32>& f, const QuantArgs& args, int64_t kb, int64_t mb,
                                                QuantRed& sm) {
  constexpr bool kRow = (kMode & kQRow) != 0;
  constexpr bool kCol = (kMode & kQCol) != 0;
  constexpr bool kBlk = (kMode & (kQBlk | kQBlkT)) != 0;
  float (&s_red)[4][128] = sm.red;
  float (&s_inv)[128] = sm.inv;
  float (&s_blkred)[4] = sm.blk;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int c = lane & 15;  // column chunk: tile columns c*8 .. c*8+7
  const int g = lane >> 4;  // row half: tile rows warp*32 + g*16 + j
  const int64_t K = args.K;
  const int64_t k0 = kb * 128;
  const int64_t m0 = mb * 128;
  const int rbase = warp * 32 + g * 16;  // tile-local first row of this thread

  // ---- 1x128 row groups ----------------------------------------------------
  if constexpr (kRow) {
    float amax[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float a = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(f.get(j, i)));
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
      amax[j] = a;
    }
    // lane c of each half computes the scale of row rbase + c ...
    float mine = amax[0];
#pragma unroll
    for (int j = 1; j < 16; ++j) mine = (c == j) ? amax[j] : mine;
    float s, inv;
    group_scale(mine, s, inv);
    const int64_t my_m = m0 + rbase + c;
    if (my_m < args.M) args.s_row[kb * args.ld_srow + my_m] = s;
    // ... and hands its inverse to the other 15 lanes of the half
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float rinv = __shfl_sync(0xffffffffu, inv, (g << 4) | j);
      const int64_t m = m0 + rbase + j;
      const uint32_t w0 = cvt_e4m3x4(f.get(j, 0) * rinv, f.get(j, 1) * rinv, f.get(j, 2) * rinv, f.get(j, 3) * rinv);
      const uint32_t w1 = cvt_e4m3x4(f.get(j, 4) * rinv, f.get(j, 5) * rinv, f.get(j, 6) * rinv, f.get(j, 7) * rinv);
      if (m < args.M) {
        *reinterpret_cast<uint2*>(args.q_row + m * K + k0 + c * 8) = make_uint2(w0, w1);
      }
    }
  }

  // ---- 128x1 column groups, stored transposed ------------------------------
  if constexpr (kCol) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float a = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) a = fmaxf(a, fabsf(f.get(j, i)));
      a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 16));
      if (g == 0) s_red[warp][c * 8 + i] = a;
    }
    __syncthreads();
    {
      const int t = threadIdx.x;  // column t of the tile
      const float a = fmaxf(fmaxf(s_red[0][t], s_red[1][t]), fmaxf(s_red[2][t], s_red[3][t]));
      float s, inv;
      group_scale(a, s, inv);
      args.s_col[mb * K + k0 + t] = s;
      s_inv[t] = inv;
    }
    __syncthreads();
    const int64_t ldT = args.M;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float cinv = s_inv[c * 8 + i];
      uint32_t w[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        w[p] = cvt_e4m3x4(f.get(4 * p + 0, i) * cinv, f.get(4 * p + 1, i) * cinv, f.get(4 * p + 2, i) * cinv,
                          f.get(4 * p + 3, i) * cinv);
      }
      *reinterpret_cast<uint4*>(args.q_colT + (k0 + c * 8 + i) * ldT + m0 + rbase) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }

  // ---- 128x128 block -------------------------------------------------------
  if constexpr (kBlk) {
    float a = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j)
#pragma unroll
      for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(f.get(j, i)));
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if (lane == 0) s_blkred[warp] = a;
    __syncthreads();
    a = fmaxf(fmaxf(s_blkred[0], s_blkred[1]), fmaxf(s_blkred[2], s_blkred[3]));
    float s, inv;
    group_scale(a, s, inv);
    const int64_t KB = K >> 7;
    const int64_t MB = args.M >> 7;
    if constexpr ((kMode & kQBlk) != 0) {
      if (threadIdx.x == 0) args.s_blk[mb * KB + kb] = s;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int64_t m = m0 + rbase + j;
        const uint32_t w0 = cvt_e4m3x4(f.get(j, 0) * inv, f.get(j, 1) * inv, f.get(j, 2) * inv, f.get(j, 3) * inv);
        const uint32_t w1 = cvt_e4m3x4(f.get(j, 4) * inv, f.get(j, 5) * inv, f.get(j, 6) * inv, f.get(j, 7) * inv);
        *reinterpret_cast<uint2*>(args.q_blk + m * K + k0 + c * 8) = make_uint2(w0, w1);
      }
    }
    if constexpr ((kMode & kQBlkT) != 0) {
      if (threadIdx.x == 0) args.s_blkT[kb * MB + mb] = s;
      const int64_t ldT = args.M;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t w[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          w[p] = cvt_e4m3x4(f.get(4 * p + 0, i) * inv, f.get(4 * p + 1, i) * inv, f.get(4 * p + 2, i) * inv,
                            f.get(4 * p + 3, i) * inv);
        }
        *reinterpret_cast<uint4*>(args.q_blkT + (k0 + c * 8 + i) * ldT + m0 + rbase) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
}

// One CTA per 128 x 128 tile (grid: K/128 x ceil(M/128)); each thread loads
// its 16 rows x 8 columns straight from global memory.  Used for FP32 input.
template <bool kF32, int kMode>
__global__ void __launch_bounds__(128) quant_tile_kernel(const QuantArgs args) {
  __shared__ QuantRed sm;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int c = lane & 15;
  const int g = lane >> 4;
  const int64_t K = args.K;
  const int64_t k0 = static_cast<int64_t>(blockIdx.x) * 128;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * 128;
  const int rbase = warp * 32 + g * 16;
  Frag<kF32> f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int64_t m = m0 + rbase + j;
    if (m < args.M) {
      const int64_t src = (args.src_rows != nullptr) ? static_cast<int64_t>(args.src_rows[m]) : m;
      f.load(args.x, src * K + k0 + c * 8, j);
    } else {
      f.zero(j);
    }
  }
  quant_tile_body<kF32, kMode>(f, args, blockIdx.x, blockIdx.y, sm);
}

// Persistent BF16 quantizer.  Each CTA walks tiles t = blockIdx.x,
// blockIdx.x + gridDim.x, ... (t -> kb = t % (K/128), mb = t / (K/128)) and
// keeps two tiles in flight: while it casts tile i from registers, tile i+1
// and, once the registers are filled, tile i+2 stream into a double-buffered
// shared-memory ring by bulk copies (one 256-byte row per thread, through an
// optional row gather).  Every thread reads its fragment out of shared
// memory (16-byte reads, two full rows per warp instruction: no bank
// conflicts).  Waits are bounded: a copy that never lands sets the status
// word, and the CTA drains what it issued and returns.
constexpr int kPipeTileBytes = 128 * 256;  // 128 rows x 128 BF16

// CTAs per SM the register budget is sized for: the two-output modes (row
// and transposed column groups, or a block with its transpose) keep more
// values live and get 2 CTAs of up to 255 registers; the others get 3.
constexpr int quant_pipe_min_blocks(int mode) {
  return (mode == (kQRow | kQCol) || mode == (kQBlk | kQBlkT)) ? 2 : 3;
}

template <int kMode>
__global__ void __launch_bounds__(128, quant_pipe_min_blocks(kMode))
    quant_pipe_kernel(const QuantArgs args, int64_t num_tiles) {
  extern __shared__ __align__(128) uint8_t qsm[];  // [2][128 rows][256 bytes]
  __shared__ QuantRed sm;
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_word;
  volatile int* abort_flag = &abort_word;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int c = lane & 15;
  const int g = lane >> 4;
  const int rbase = warp * 32 + g * 16;
  const int64_t K = args.K;
  const int64_t kbt = K >> 7;
  const uint32_t bar0 = smem_u32(&bars[0]);
  const uint32_t buf0 = smem_u32(qsm);

  // bytes that land in the buffer for tile tt (rows past M are not copied)
  auto tile_bytes = [&](int64_t tt) -> uint32_t {
    const int64_t rows = args.M - (tt / kbt) * 128;
    return static_cast<uint32_t>(rows < 128 ? rows : 128) * 256u;
  };
  // this thread's row copy of tile tt into buffer b
  auto issue_row = [&](int64_t tt, int b) {
    const int64_t m = (tt / kbt) * 128 + tid;
    if (m < args.M) {
      const int64_t src = (args.src_rows != nullptr) ? static_cast<int64_t>(args.src_rows[m]) : m;
      bulk_load(buf0 + b * kPipeTileBytes + tid * 256,
                static_cast<const uint16_t*>(args.x) + src * K + (tt % kbt) * 128, 256u, bar0 + 8 * b);
    }
  };

  if (tid == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8, 1);
    abort_word = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int64_t t0 = blockIdx.x, t1 = blockIdx.x + gridDim.x;
  if (tid == 0) {
    if (t0 < num_tiles) mbar_arrive_expect_tx(bar0, tile_bytes(t0));
    if (t1 < num_tiles) mbar_arrive_expect_tx(bar0 + 8, tile_bytes(t1));
  }
  __syncthreads();
  if (t0 < num_tiles) issue_row(t0, 0);
  if (t1 < num_tiles) issue_row(t1, 1);

  uint32_t it = 0;
  int64_t t = t0;
  for (; t < num_tiles; t += gridDim.x, ++it) {
    const int b = it & 1;
    const bool ok = mbar_wait(bar0 + 8 * b, (it >> 1) & 1u, abort_flag);
    Frag<false> f;
    if (ok) {
      const uint8_t* tile = qsm + b * kPipeTileBytes;
#pragma unroll
      for (int j = 0; j < 16; ++j) f.v[j] = *reinterpret_cast<const uint4*>(tile + (rbase + j) * 256 + c * 16);
    }
    const int64_t tn = t + 2 * static_cast<int64_t>(gridDim.x);
    if (ok && tid == 0 && tn < num_tiles) mbar_arrive_expect_tx(bar0 + 8 * b, tile_bytes(tn));
    // every thread has its fragment (buffer b is free) or some wait failed
    if (__syncthreads_or(!ok)) break;
    if (tn < num_tiles) issue_row(tn, b);
    // rows past M were not copied: their registers hold stale data, but
    // quant_tile_body neither stores nor reduces rows >= M
    quant_tile_body<false, kMode>(f, args, t % kbt, t / kbt, sm);
  }
  // the code tiles' stores have completed before the CTA exits
  if (tid == 0 || tid == 128) bulk_wait_all();
  if (t < num_tiles) {
    // a wait failed: let every copy this CTA issued land before it exits
    // (bounded; the status word already records the timeout)
    for (uint32_t d = 0; d < 2; ++d) {
      const uint32_t u = it + d;  // iteration whose copy may be in flight
      if (t + static_cast<int64_t>(d) * gridDim.x >= num_tiles) break;
      const uint64_t s0 = globaltimer_ns();
      while (!mbar_try_wait(bar0 + 8 * (u & 1u), (u >> 1) & 1u) && globaltimer_ns() - s0 < 1000000ull) {}
    }
  }
}

// ---------------------------------------------------------------------------
// BF16 tiles through TMA, split by role: row groups and/or transposed column
// groups of activations, or (kBlk) a 128x128 block's codes as-is and/or
// transposed.  Persistent, 128 threads per path present, two 128 x 128 tiles
// in flight per CTA, each arriving as one dense TMA box (128 rows x 256 bytes).
//   row path     thread r owns tile row r (16 x 16-byte reads, in a rotated
//                order that keeps them free of bank conflicts); its 1x128
//                amax is a packed BF16 max over the row (no shuffles).
//   column path  thread (p, h) owns columns 2p, 2p+1 over the 64 rows of
//                half h (64 x 4-byte reads); the two halves meet in shared
//                memory for the 128x1 amax.
// In block mode each path holds the whole tile, so each finds the block's
// amax by itself (warp shuffles, then its 4 warps' maxima in shared memory)
// and casts with that one scale: the row path writes the codes as they lie,
// the column path their transpose.
// Each path writes its 128 x 128 codes into a staged shared-memory tile in
// the 128-byte-swizzled layout (16-byte chunk c of row r at chunk c ^ (r % 8),
// which keeps those writes conflict-free) and one thread stores the tile
// with a single TMA store (whole lines; rows past M are clipped).  The store
// must have read the tile before the next tile is staged: its issuer waits
// for that just before the CTA barrier every tile passes anyway.  The amax
// is exact in BF16; the scale and cast are those of quant_tile_body.
// ---------------------------------------------------------------------------
constexpr int kRcPitch = 256;                 // bytes per smem tile row (one dense TMA box)
constexpr int kRcTileBytes = 128 * kRcPitch;  // one tile buffer
constexpr int kRcCodePitch = 128;             // bytes per row of a staged (swizzled) 128 x 128 code tile
constexpr int kRcCodeBytes = 128 * kRcCodePitch;
constexpr int kRcSmem = 2 * kRcTileBytes + 2 * kRcCodeBytes;  // inputs, row codes, transposed codes


// Shared memory of quant_rc_kernel<kRow, kCol>: two input tiles, then one
// staged code tile per path (+ slack to align the base to 1024 bytes, the
// 128-byte swizzle's period; the tile buffers are multiples of 1024 bytes).
constexpr int rc_smem_bytes(bool row, bool col) {
  return 2 * kRcTileBytes + ((row ? 1 : 0) + (col ? 1 : 0)) * kRcCodeBytes + 1024;
}
static_assert(kRcTileBytes % 1024 == 0 && kRcCodeBytes % 1024 == 0, "staged tiles must stay 1024-aligned");

template <bool kRow, bool kCol, bool kBlk, bool kMx = false>
__global__ void __launch_bounds__((kRow ? 128 : 0) + (kCol ? 128 : 0), 2)
    quant_rc_kernel(const QuantArgs args, int64_t num_tiles, const __grid_constant__ CUtensorMap tm_x,
                    const __grid_constant__ CUtensorMap tm_row, const __grid_constant__ CUtensorMap tm_col) {
  extern __shared__ __align__(128) uint8_t rsm_raw[];
  // [2][128][kRcPitch] inputs, then the staged code tiles
  uint8_t* rsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rsm_raw) + 1023) & ~uintptr_t(1023));
  __shared__ float s_cmax[2][128];                 // column maxima of each 64-row half
  __shared__ float s_bmax[2][4];                   // block mode: per-warp maxima of each path
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_word;
  volatile int* abort_flag = &abort_word;

  const int tid = threadIdx.x;
  const int64_t K = args.K;
  const int64_t M = args.M;
  const int64_t kbt = K >> 7;
  const uint32_t bar0 = smem_u32(&bars[0]);
  const uint32_t buf0 = smem_u32(rsm);

  // Input tile tt: one TMA load of 128 rows x 128 columns (256-byte rows,
  // dense, no swizzle).  The row path reads its row's 16-byte chunks in a
  // rotated order, which keeps those reads free of bank conflicts.
  static_assert(kRow || kCol, "at least one path");
  static_assert(!kMx || (kRow && !kCol && !kBlk), "MX groups: the row path alone");
  auto tile_bytes = [&](int64_t) -> uint32_t { return static_cast<uint32_t>(kRcTileBytes); };
  auto issue_tile = [&](int64_t tt, int b) {  // one thread
    tma_load_2d(buf0 + b * kRcTileBytes, &tm_x, static_cast<int32_t>((tt % kbt) * 128),
                static_cast<int32_t>((tt / kbt) * 128), bar0 + 8 * b);
  };
  // the row path runs on threads 0..127; the column path on the next 128
  // (or on 0..127 when it is alone)
  const bool row_role = kRow && (!kCol || tid < 128);
  const int ctid = kRow ? tid - 128 : tid;

  if (tid == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8, 1);
    abort_word = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int64_t t0 = blockIdx.x, t1 = blockIdx.x + gridDim.x;
  if (tid == 0) {
    if (t0 < num_tiles) {
      mbar_arrive_expect_tx(bar0, tile_bytes(t0));
      issue_tile(t0, 0);
    }
    if (t1 < num_tiles) {
      mbar_arrive_expect_tx(bar0 + 8, tile_bytes(t1));
      issue_tile(t1, 1);
    }
  }

  uint32_t it = 0;
  int64_t t = t0;
  for (; t < num_tiles; t += gridDim.x, ++it) {
    const int b = it & 1;
    const bool ok = mbar_wait(bar0 + 8 * b, (it >> 1) & 1u, abort_flag);
    const uint8_t* tile = rsm + b * kRcTileBytes;
    const int64_t kb = t % kbt, mb = t / kbt;
    const int64_t k0 = kb * 128, m0 = mb * 128;
    // one register array for either path (the paths are warp-uniform, so
    // only one of them is ever live): row path, the row's 128 values as 16
    // x 4 words; column path, columns 2p, 2p+1 of 64 rows, one word each
    uint32_t w[64];
    const int p = ctid & 63;
    const int hh = ctid >> 6;
    if (ok) {
      if (row_role) {
        // slot k (words 8k .. 8k+7) holds code chunk (k + tid) % 8, i.e. input
        // chunks 2((k + tid) % 8) and +1; threads with (tid / 8) odd read the
        // odd chunk of the pair first.  Each 16-byte read then spreads 32
        // threads evenly over the 8 bank groups.
        const uint8_t* rp = tile + tid * kRcPitch;
        const int r8 = tid & 7, s8 = (tid >> 3) & 1;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int kk = (k + r8) & 7;
          const uint4 qa = *reinterpret_cast<const uint4*>(rp + (2 * kk + s8) * 16);
          const uint4 qb = *reinterpret_cast<const uint4*>(rp + (2 * kk + 1 - s8) * 16);
          const uint4 lo = s8 ? qb : qa, hi = s8 ? qa : qb;
          w[8 * k] = lo.x;
          w[8 * k + 1] = lo.y;
          w[8 * k + 2] = lo.z;
          w[8 * k + 3] = lo.w;
          w[8 * k + 4] = hi.x;
          w[8 * k + 5] = hi.y;
          w[8 * k + 6] = hi.z;
          w[8 * k + 7] = hi.w;
        }
      } else {
        const uint8_t* cp = tile + (hh * 64) * kRcPitch + p * 4;
#pragma unroll
        for (int r = 0; r < 64; ++r) w[r] = *reinterpret_cast<const uint32_t*>(cp + r * kRcPitch);
      }
    }
    const int64_t tn = t + 2 * static_cast<int64_t>(gridDim.x);
    if (ok && tid == 0 && tn < num_tiles) mbar_arrive_expect_tx(bar0 + 8 * b, tile_bytes(tn));
    // each path's store issuer: the previous tile's store has read its staged codes
    if (tid == 0 || tid == 128) bulk_wait_read<0>();
    // every thread has its values (buffer b is free), the staged code tiles
    // are free, or some wait failed
    if (__syncthreads_or(!ok)) break;
    if (tid == 0 && tn < num_tiles) issue_tile(tn, b);

    if (row_role) {
      const int64_t m = m0 + tid;
      if constexpr (kMx) {
        // ---- MX: four 1x32 groups of row m.  Slot k holds code chunk
        // j = (k + tid) % 8 (16 columns), which belongs to group j / 2.
        float gmax[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          __nv_bfloat162 h = __habs2(bf2_of(w[8 * k]));
#pragma unroll
          for (int i = 1; i < 8; ++i) h = __hmax2(h, __habs2(bf2_of(w[8 * k + i])));
          const uint32_t hw = u32_of(h);
          const float a = fmaxf(bf16lo_to_f32(hw), bf16hi_to_f32(hw));
          const int g = ((k + tid) & 7) >> 1;
#pragma unroll
          for (int gg = 0; gg < 4; ++gg) gmax[gg] = g == gg ? fmaxf(gmax[gg], a) : gmax[gg];
        }
        uint32_t word = 0;
        float ginv[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const uint32_t byte = mx_scale_byte(gmax[g]);
          ginv[g] = __uint_as_float((254u - byte) << 23);  // 2^-(byte - 127), a normal float
          word |= byte << (8 * g);
        }
        // rows past the end get scale 1 (byte 127): defined, never read into C
        const int64_t rt_count = (M + 127) >> 7;
        *reinterpret_cast<uint32_t*>(args.s_mx + (kb * rt_count + mb) * 512 + (tid & 31) * 16 + (tid >> 5) * 4) =
            m < M ? word : 0x7F7F7F7Fu;
        uint4* st = reinterpret_cast<uint4*>(rsm + 2 * kRcTileBytes + tid * kRcCodePitch);  // row tid
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int g = ((k + tid) & 7) >> 1;
          const float inv = g == 0 ? ginv[0] : g == 1 ? ginv[1] : g == 2 ? ginv[2] : ginv[3];
          uint32_t c[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t a = w[8 * k + 2 * u], bb = w[8 * k + 2 * u + 1];
            c[u] = cvt_e4m3x4(bf16lo_to_f32(a) * inv, bf16hi_to_f32(a) * inv, bf16lo_to_f32(bb) * inv,
                              bf16hi_to_f32(bb) * inv);
          }
          st[((k + tid) & 7) ^ (tid & 7)] = make_uint4(c[0], c[1], c[2], c[3]);  // code chunk of slot k
        }
        fence_proxy_async_smem();
        asm volatile("bar.sync 3, 128;" ::: "memory");
        if (tid == 0) {
          tma_store_2d(&tm_row, smem_u32(rsm + 2 * kRcTileBytes), static_cast<int32_t>(k0),
                       static_cast<int32_t>(m0));
          bulk_commit();
        }
      } else {
        // ---- 1x128 row group of row m
        __nv_bfloat162 mx = __habs2(bf2_of(w[0]));
#pragma unroll
        for (int i = 1; i < 64; ++i) mx = __hmax2(mx, __habs2(bf2_of(w[i])));
        const uint32_t mw = u32_of(mx);
        float amax = fmaxf(bf16lo_to_f32(mw), bf16hi_to_f32(mw));
        if constexpr (kBlk) {
          // the 128x128 block's amax: over the warp, then over the path's 4 warps
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
          if ((tid & 31) == 0) s_bmax[0][tid >> 5] = amax;
          asm volatile("bar.sync 3, 128;" ::: "memory");
          amax = fmaxf(fmaxf(s_bmax[0][0], s_bmax[0][1]), fmaxf(s_bmax[0][2], s_bmax[0][3]));
        }
        float sc, inv;
        group_scale(amax, sc, inv);
        if constexpr (kBlk) {
          if (tid == 0) args.s_blk[mb * kbt + kb] = sc;
        } else {
          if (m < M) args.s_row[kb * args.ld_srow + m] = sc;
        }
        uint4* st = reinterpret_cast<uint4*>(rsm + 2 * kRcTileBytes + tid * kRcCodePitch);  // row tid
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          uint32_t c[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t a = w[4 * i + 2 * u], bb = w[4 * i + 2 * u + 1];
            c[u] = cvt_e4m3x4(bf16lo_to_f32(a) * inv, bf16hi_to_f32(a) * inv, bf16lo_to_f32(bb) * inv,
                              bf16hi_to_f32(bb) * inv);
          }
          st[(((i >> 1) + tid) & 7) ^ (tid & 7)] = make_uint4(c[0], c[1], c[2], c[3]);  // code chunk of slot i/2
        }
        fence_proxy_async_smem();
        asm volatile("bar.sync 3, 128;" ::: "memory");
        if (tid == 0) {
          tma_store_2d(&tm_row, smem_u32(rsm + 2 * kRcTileBytes), static_cast<int32_t>(k0), static_cast<int32_t>(m0));
          bulk_commit();
        }
      }
    } else if constexpr (kCol) {
      // ---- 128x1 column groups of columns k0 + 2p, k0 + 2p + 1
      __nv_bfloat162 mx = __habs2(bf2_of(w[0]));
#pragma unroll
      for (int r = 1; r < 64; ++r) mx = __hmax2(mx, __habs2(bf2_of(w[r])));
      const uint32_t mw = u32_of(mx);
      float sc0, inv0, sc1, inv1;
      if constexpr (kBlk) {
        // the 128x128 block's amax: over the warp, then over the path's 4 warps
        float amax = fmaxf(bf16lo_to_f32(mw), bf16hi_to_f32(mw));
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if ((ctid & 31) == 0) s_bmax[1][ctid >> 5] = amax;
        asm volatile("bar.sync 2, 128;" ::: "memory");
        amax = fmaxf(fmaxf(s_bmax[1][0], s_bmax[1][1]), fmaxf(s_bmax[1][2], s_bmax[1][3]));
        group_scale(amax, sc0, inv0);
        sc1 = sc0;
        inv1 = inv0;
        if (ctid == 0) args.s_blkT[kb * (M >> 7) + mb] = sc0;
      } else {
        s_cmax[hh][2 * p] = bf16lo_to_f32(mw);
        s_cmax[hh][2 * p + 1] = bf16hi_to_f32(mw);
        asm volatile("bar.sync 2, 128;" ::: "memory");
        group_scale(fmaxf(s_cmax[0][2 * p], s_cmax[1][2 * p]), sc0, inv0);
        group_scale(fmaxf(s_cmax[0][2 * p + 1], s_cmax[1][2 * p + 1]), sc1, inv1);
        if (hh == 0) *reinterpret_cast<float2*>(args.s_col + mb * K + k0 + 2 * p) = make_float2(sc0, sc1);
      }
      // staged transposed tile: row = column of x, 128 token bytes per row
      uint8_t* ct = rsm + 2 * kRcTileBytes + (kRow ? kRcCodeBytes : 0);
      uint4* d0 = reinterpret_cast<uint4*>(ct + (2 * p) * kRcCodePitch);
      uint4* d1 = reinterpret_cast<uint4*>(ct + (2 * p + 1) * kRcCodePitch);
#pragma unroll
      for (int r = 0; r < 64; r += 16) {
        uint32_t c0[4], c1[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t a = w[r + 4 * u], bb = w[r + 4 * u + 1], cc = w[r + 4 * u + 2], dd = w[r + 4 * u + 3];
          c0[u] = cvt_e4m3x4(bf16lo_to_f32(a) * inv0, bf16lo_to_f32(bb) * inv0, bf16lo_to_f32(cc) * inv0,
                             bf16lo_to_f32(dd) * inv0);
          c1[u] = cvt_e4m3x4(bf16hi_to_f32(a) * inv1, bf16hi_to_f32(bb) * inv1, bf16hi_to_f32(cc) * inv1,
                             bf16hi_to_f32(dd) * inv1);
        }
        // token chunk hh * 4 + r / 16 of rows 2p and 2p+1, swizzled
        d0[(hh * 4 + (r >> 4)) ^ ((2 * p) & 7)] = make_uint4(c0[0], c0[1], c0[2], c0[3]);
        d1[(hh * 4 + (r >> 4)) ^ ((2 * p + 1) & 7)] = make_uint4(c1[0], c1[1], c1[2], c1[3]);
      }
      fence_proxy_async_smem();
      asm volatile("bar.sync 2, 128;" ::: "memory");
      if (ctid == 0) {
        tma_store_2d(&tm_col, smem_u32(ct), static_cast<int32_t>(m0), static_cast<int32_t>(k0));
        bulk_commit();
      }
    }
  }
  // the code tiles' stores have completed before the CTA exits
  if (tid == 0 || tid == 128) bulk_wait_all();
  if (t < num_tiles) {
    // a wait failed: let every copy this CTA issued land before it exits
    for (uint32_t d = 0; d < 2; ++d) {
      const uint32_t u = it + d;
      if (t + static_cast<int64_t>(d) * gridDim.x >= num_tiles) break;
      const uint64_t s0 = globaltimer_ns();
      while (!mbar_try_wait(bar0 + 8 * (u & 1u), (u >> 1) & 1u) && globaltimer_ns() - s0 < 1000000ull) {}
    }
  }
}


}  // namespace fp8q
