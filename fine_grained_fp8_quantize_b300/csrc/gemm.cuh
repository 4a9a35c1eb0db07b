// gemm.cuh -- block-scaled FP8 (E4M3) GEMM with FP32 promotion every 128 K,
// dense and MoE-grouped, for sm_103a (tcgen05 + TMEM + TMA).
//
// The method: tensor cores accumulate each 128-element K interval with their
// own limited internal precision; at the end of the interval the partial sum
// is copied to FP32 registers on the CUDA cores, multiplied by the two
// dequantization scales and added into a full-precision FP32 accumulator
// ("Eliminate Deepseek Ai News For Good", the MMA-precision passage;
// inprokorea.com page, the 128-element accumulation-interval passage;
// "Is aI Hitting a Wall?", the dequantization passage).
//
// B300 design (the pages' Hopper ping-pong of two WGMMA warpgroups is prior
// art, replaced by):
//   warp 0       TMA producer: one 128x128 A tile + one 256x128 B tile per
//                K-block into a kStages-deep ring of 128B-swizzled smem.
//   warp 1       MMA issuer and TMEM owner: per K-block four
//                tcgen05.mma.kind::f8f6f4 (128x256x32) into a FRESH TMEM
//                partial (the first with accumulate off).  Two partial
//                buffers (2 x 256 FP32 columns = all 512) alternate, so the
//                MMAs of block kb+1 overlap the promotion of block kb.
//                Warps 0 and 1 run their loops as whole warps and issue from
//                one elected lane, which keeps the operands warp-uniform.
//   warp 2       scale warp (variants with the scale ring): copies each
//                K-block's A and B scales into a shared-memory ring ahead of
//                use, a batch of K-blocks per slot (see the ring below).
//   warps 4..11  promotion + epilogue: each thread owns one row and 128
//                columns of the 128x256 tile in 128 FP32 registers; per
//                K-block it tcgen05.ld's its slice of the partial, frees the
//                buffer, and does acc = fma(P, sA*sB, acc).  At the end of
//                a tile it rounds (BF16, RNE) or keeps FP32 and stores.
// Registers: warpgroup 0 gives up all but 56 (ring variants: 40) per
// thread (setmaxnreg) so the two promotion warpgroups can hold 224 (232)
// each: the 384 x 168 registers of the launch, exactly.
// The grid is persistent (one CTA per SM); tiles are striped over CTAs,
// M-tile fastest (in groups of M-tiles when A is large), and a stream-K
// variant splits the last waves' tiles by K over all CTAs.
// Every mbarrier wait is bounded (see mbar_wait): on expiry the kernel
// records a timeout in the status word and unwinds without trapping.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "ptx.cuh"

namespace fp8q {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 128;
constexpr int kStages = 4;
constexpr int kGemmThreads = 384;
// Register split after setmaxnreg, warpgroup 0 (producer, MMA issuer, scale
// warp, one idle warp) / warpgroups 1-2 (promotion).  Both add up to the
// launch's 384 x 168 (128 x ctl + 256 x math; setmaxnreg.inc may not ask for
// more).  The ring variants keep more state in the promotion warps and give
// them 232; the others measured best at 56 / 224.
__host__ __device__ constexpr uint32_t regs_ctl(bool ring) { return ring ? 40u : 56u; }
__host__ __device__ constexpr uint32_t regs_math(bool ring) { return ring ? 232u : 224u; }
static_assert(128 * regs_ctl(false) + 256 * regs_math(false) <= 384 * 168 &&
                  128 * regs_ctl(true) + 256 * regs_math(true) <= 384 * 168,
              "register split over the launch's 384 x 168");
constexpr int kMaxExperts = 1024;
constexpr uint32_t kABytes = kBM * kBK;  // 16 KB
constexpr uint32_t kBBytes = kBN * kBK;  // 32 KB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdesc = idesc_e4m3_f32(kBM, kBN);

// Scale ring.  A dedicated warp copies every K-block's scales into shared
// memory ahead of use: the A scales of rows a0 .. a0+131 (a0 = the tile's
// first row rounded down to a multiple of 4, so one bulk copy starts
// 16-byte aligned), then the B scales (the two 128x128-block scales of the
// tile's column halves, or its 256 per-column scales).  Slots hold a batch
// of consecutive K-blocks, so the promotion warps wait for a slot and
// release it once per batch and otherwise read plain shared memory.
// A slot is refilled (kScR - 1) batches before it is read: per-column
// entries are large (1.5 KB a K-block), so they come two K-blocks a batch
// in four slots, which measured faster than four in two slots (less lead)
// and one in eight (a barrier round per K-block).
constexpr uint32_t kScRowBytes = 132 * 4 + 16;
__host__ __device__ constexpr uint32_t sc_kb_bytes(int sb_gran) { return kScRowBytes + (sb_gran == 1 ? kBN * 4 : 16); }
__host__ __device__ constexpr int sc_batch(int sb_gran) { return sb_gran == 1 ? 2 : 8; }
__host__ __device__ constexpr int sc_ring(int sb_gran, bool grouped) { return sb_gran == 1 ? 4 : (grouped ? 2 : 4); }
__host__ __device__ constexpr uint32_t sc_slot_bytes(int sb_gran) { return sc_batch(sb_gran) * sc_kb_bytes(sb_gran); }

// dynamic shared memory layout (offsets from a 1024-aligned base)
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + kStages * kABytes;
constexpr uint32_t kChunkBytes = 32 * 32;                // epilogue chunk: 32 rows x 32 bytes
constexpr uint32_t kOffSc = kOffB + kStages * kBBytes;  // scale ring
// epilogue staging, 2 chunks per warp: the source of TMA tensor stores, so
// 128-byte aligned
__host__ __device__ constexpr uint32_t off_stage(int g, bool grp) {
  return (kOffSc + sc_ring(g, grp) * sc_slot_bytes(g) + 127u) & ~127u;
}
__host__ __device__ constexpr uint32_t off_bar(int g, bool grp) { return off_stage(g, grp) + 8 * 2 * kChunkBytes; }
__host__ __device__ constexpr uint32_t off_misc(int g, bool grp) { return off_bar(g, grp) + 48 * 8; }  // tmem base, abort
__host__ __device__ constexpr uint32_t off_pref(int g, bool grp) { return off_misc(g, grp) + 16; }  // grouped: [E+1]
__host__ __device__ constexpr uint32_t off_rowoff(int g, bool grp) { return off_pref(g, grp) + 4 * (kMaxExperts + 1); }
__host__ __device__ constexpr uint32_t gemm_smem_bytes(int g, bool grp) {
  return (grp ? off_rowoff(g, grp) + 4 * (kMaxExperts + 1) : off_pref(g, grp)) + 1024;  // + alignment slack
}
static_assert(off_stage(128, false) % 128 == 0 && off_stage(128, true) % 128 == 0 && off_stage(1, false) % 128 == 0,
              "TMA store sources must be 128-byte aligned");
static_assert(sc_slot_bytes(128) % 16 == 0 && sc_slot_bytes(1) % 16 == 0 && sc_kb_bytes(128) % 16 == 0 &&
                  sc_kb_bytes(1) % 16 == 0,
              "bulk copies into the scale ring need 16-byte aligned destinations");
static_assert(gemm_smem_bytes(128, false) <= 232448 && gemm_smem_bytes(128, true) <= 232448 &&
                  gemm_smem_bytes(1, false) <= 232448,
              "GEMM shared memory over the 227 KB per-CTA limit");

struct GemmArgs {
  const float* sA;   // [K/128][lds_a]
  int64_t lds_a;
  const float* sB;   // gran 128: [E][N/128][K/128]; gran 1: [K/128][N]
  void* C;           // [rows][N]
  int64_t M;         // dense rows
  int64_t N;
  int64_t K;
  int tiles_m;       // dense
  int tiles_n;
  int m_group;       // dense: M-tiles per raster group (tiles_m: plain M-fastest order)
  const int32_t* row_offsets;  // grouped [E+1]
  int E;
  // stream-K (dense only, kernel variant kStreamK): tiles below sk_tile0 are
  // whole tiles striped over the CTAs (data-parallel waves, which keep
  // concurrently running CTAs on neighbouring tiles); each CTA then takes
  // an equal share of the tile-major sequence of the remaining tiles'
  // K-blocks.  A tile split between CTAs is finished by the CTA holding its
  // first K-blocks, which adds the other CTAs' FP32 partial tiles (ws, slot
  // = CTA index) once their flags carry this call's epoch.
  int streamk;
  int sk_tile0;
  // 1 when every K-block's A scales can be fetched with one bulk copy
  // (lds_a and M multiples of 4); else the scale warp's lanes copy them
  int sa_bulk;
  float4* ws;        // [gridDim.x][2 halves][32 column quads][128 rows] float4
  uint32_t* flags;   // [gridDim.x], zero between calls
  uint32_t epoch;    // nonzero, distinct from the previous call's
};

// First K-block of CTA `cta` of `grid` in the stream-K split of `total`
// K-blocks (CTA c takes [begin(c), begin(c+1))).
__device__ __forceinline__ int64_t streamk_begin(int64_t total, int64_t cta, int64_t grid) {
  return total * cta / grid;
}

// This CTA's work as segments (tile t, K-blocks [lo, hi)): the tiles
// t = blockIdx.x + i * gridDim.x below the stream-K start (whole tiles),
// then, in the stream-K variant, its equal share of the K-blocks of the
// tiles from a.sk_tile0 on.  f(t, lo, hi) returns false to stop.
template <bool kStreamK, typename F>
__device__ __forceinline__ void for_each_segment(const GemmArgs& a, int num_tiles, int64_t KB, F&& f) {
  const int dp_end = kStreamK ? a.sk_tile0 : num_tiles;
  for (int t = blockIdx.x; t < dp_end; t += gridDim.x)
    if (!f(t, int64_t(0), KB)) return;
  if constexpr (kStreamK) {
    const int64_t all = static_cast<int64_t>(num_tiles - a.sk_tile0) * KB;
    const int64_t e = streamk_begin(all, static_cast<int64_t>(blockIdx.x) + 1, gridDim.x);
    for (int64_t it = streamk_begin(all, blockIdx.x, gridDim.x); it < e;) {
      const int tr = static_cast<int>(it / KB);
      const int64_t lo = it - static_cast<int64_t>(tr) * KB;
      const int64_t hi = e - static_cast<int64_t>(tr) * KB < KB ? e - static_cast<int64_t>(tr) * KB : KB;
      if (!f(a.sk_tile0 + tr, lo, hi)) return;
      it += hi - lo;
    }
  }
}

// K-blocks of all of this CTA's segments.
template <bool kStreamK>
__device__ __forceinline__ uint64_t cta_kblocks(const GemmArgs& a, int num_tiles, int64_t KB) {
  const int dp_end = kStreamK ? a.sk_tile0 : num_tiles;
  const int64_t local_tiles =
      static_cast<int>(blockIdx.x) < dp_end ? (dp_end - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
  uint64_t total = static_cast<uint64_t>(local_tiles) * static_cast<uint64_t>(KB);
  if constexpr (kStreamK) {
    const int64_t all = static_cast<int64_t>(num_tiles - a.sk_tile0) * KB;
    total += static_cast<uint64_t>(streamk_begin(all, static_cast<int64_t>(blockIdx.x) + 1, gridDim.x) -
                                   streamk_begin(all, blockIdx.x, gridDim.x));
  }
  return total;
}

struct TileInfo {
  int64_t m0;       // first row (global)
  int64_t row_end;  // rows >= row_end are not this tile's
  int64_t n0;       // first column
  int32_t b_row;    // row coordinate of the B tile in the B tensor map
  int64_t sb_off;   // expert offset into sB (grouped)
};

template <bool kGrouped>
__device__ __forceinline__ TileInfo tile_info(int t, const GemmArgs& a, const int* pref, const int* roff) {
  TileInfo ti;
  if constexpr (!kGrouped) {
    // groups of m_group M-tiles, each over all N-tiles, M-fastest inside
    const int per = a.m_group * a.tiles_n;
    const int grp = t / per;
    const int w = t - grp * per;
    const int m_lo = grp * a.m_group;
    const int gm = a.tiles_m - m_lo < a.m_group ? a.tiles_m - m_lo : a.m_group;
    const int mt = m_lo + w % gm;
    const int nt = w / gm;
    ti.m0 = static_cast<int64_t>(mt) * kBM;
    ti.row_end = a.M;
    ti.n0 = static_cast<int64_t>(nt) * kBN;
    ti.b_row = nt * kBN;
    ti.sb_off = 0;
  } else {
    // expert e with pref[e] <= t < pref[e+1] (largest such e skips empties)
    int lo = 0, hi = a.E;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pref[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int r0 = roff[e], r1 = roff[e + 1];
    const int mtiles = (r1 - r0 + kBM - 1) / kBM;
    const int local = t - pref[e];
    const int nt = local / mtiles;  // all M-tiles of one N-slab run together
    const int mt = local % mtiles;
    ti.m0 = r0 + static_cast<int64_t>(mt) * kBM;
    ti.row_end = r1 < a.M ? r1 : a.M;  // never past total_rows, even for bad offsets
    ti.n0 = static_cast<int64_t>(nt) * kBN;
    ti.b_row = static_cast<int32_t>(static_cast<int64_t>(e) * a.N + ti.n0);
    ti.sb_off = static_cast<int64_t>(e) * (a.N / 128) * (a.K / 128);
  }
  return ti;
}

// kRing: scales through the shared-memory ring (required for per-column B
// scales and the grouped form); else loaded by the promotion warps.
template <bool kOutF32, int kSbGran, bool kGrouped, bool kStreamK, bool kRing>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  constexpr int kScB = sc_batch(kSbGran);              // K-blocks per scale slot
  constexpr int kScR = sc_ring(kSbGran, kGrouped);     // scale slots
  constexpr uint32_t kScKb = sc_kb_bytes(kSbGran);
  constexpr uint32_t kScSlot = sc_slot_bytes(kSbGran);
  constexpr uint32_t kOffStage = off_stage(kSbGran, kGrouped);
  const uint32_t bar_full = sbase + off_bar(kSbGran, kGrouped);  // [kStages]
  const uint32_t bar_empty = bar_full + kStages * 8;    // [kStages]
  const uint32_t bar_tfull = bar_empty + kStages * 8;   // [2]
  const uint32_t bar_tempty = bar_tfull + 2 * 8;        // [2]
  const uint32_t bar_drain = bar_tempty + 2 * 8;        // [1]
  const uint32_t bar_sfull = bar_drain + 8;             // [kScR]
  const uint32_t bar_sempty = bar_sfull + kScR * 8;     // [kScR]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + off_misc(kSbGran, kGrouped));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + off_misc(kSbGran, kGrouped) + 4);
  int* pref = reinterpret_cast<int*>(smem + off_pref(kSbGran, kGrouped));
  int* roff = reinterpret_cast<int*>(smem + off_rowoff(kSbGran, kGrouped));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t KB = args.K / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, 8);  // one arrive per promotion warp
    }
    mbar_init(bar_drain, 1);
    for (int r = 0; r < kScR; ++r) {
      mbar_init(bar_sfull + 8 * r, 1);   // the scale warp's arrival at the end of a batch (+ its copies' bytes)
      mbar_init(bar_sempty + 8 * r, 8);  // one arrive per promotion warp
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if constexpr (kGrouped) {
    if (warp == 4) {
      // tile prefix over experts: pref[e] = sum_{e' < e} ceil(rows_e'/128) * tiles_n
      const int E = args.E;
      const int per = (E + 31) / 32;
      const int lo = lane * per;
      const int hi = min(E, lo + per);
      int local = 0;
      for (int e = lo; e < hi; ++e) {
        const int r0 = __ldg(args.row_offsets + e), r1 = __ldg(args.row_offsets + e + 1);
        roff[e] = r0;
        local += ((r1 - r0 + kBM - 1) / kBM) * args.tiles_n;
      }
      int incl = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int run = incl - local;
      for (int e = lo; e < hi; ++e) {
        pref[e] = run;
        const int r0 = roff[e], r1 = __ldg(args.row_offsets + e + 1);
        run += ((r1 - r0 + kBM - 1) / kBM) * args.tiles_n;
      }
      if (lane == 31) {
        pref[E] = incl;
        roff[E] = __ldg(args.row_offsets + E);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int num_tiles = kGrouped ? pref[args.E] : args.tiles_m * args.tiles_n;

  if (warp < 4) {
    setmaxnreg_dec<regs_ctl(kRing)>();
  }
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // the whole warp runs the loop; one elected lane issues the copies
    {
      uint32_t stage = 0, phase = 0, issued = 0;
      bool ok = true;
      // K-blocks [kb_lo, kb_hi) of tile t
      auto load_tile = [&](int t, int64_t kb_lo, int64_t kb_hi) {
        const TileInfo ti = tile_info<kGrouped>(t, args, pref, roff);
        for (int64_t kb = kb_lo; kb < kb_hi; ++kb) {
          if (!mbar_wait_warp(bar_empty + 8 * stage, phase ^ 1u, abort_flag)) { ok = false; break; }
          if (elect_one()) {
            mbar_arrive_expect_tx(bar_full + 8 * stage, kABytes + kBBytes);
            tma_load_2d(sbase + kOffA + stage * kABytes, &tmA, static_cast<int32_t>(kb * kBK),
                        static_cast<int32_t>(ti.m0), bar_full + 8 * stage);
            tma_load_2d(sbase + kOffB + stage * kBBytes, &tmB, static_cast<int32_t>(kb * kBK), ti.b_row,
                        bar_full + 8 * stage);
          }
          __syncwarp();
          ++issued;
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      };
      for_each_segment<kStreamK>(args, num_tiles, KB, [&](int t, int64_t lo, int64_t hi) {
        load_tile(t, lo, hi);
        return ok;
      });
      if (!ok && lane == 0) {
        // drain: wait (bounded) for the copies still in flight
        for (uint32_t i = 0; i < kStages && i < issued; ++i) {
          if (stage == 0) { stage = kStages; phase ^= 1u; }
          --stage;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(bar_full + 8 * stage, phase) && globaltimer_ns() - t0 < 1000000ull) {}
        }
      }
    }
  } else if (kRing && warp == 2) {
    // ------------------------------------------------------------ scale warp
    // Fills the scale ring batch by batch, as far ahead as it has free slots
    // (a slot is free once the promotion warps have read its last K-block),
    // independently of the operand stages: the scales' global-load latency
    // hides behind many K-blocks.  Per K-block, A's row scales are one bulk
    // copy when aligned (else the lanes copy them); the two block scales of
    // B come from registers the warp loaded once per tile (lanes 0 and 1
    // store them); per-column B scales are a second bulk copy.  The slot's
    // full barrier gets the bytes of each copy (expect_tx) and one arrival
    // at the end of the batch.
    {
      uint32_t g = 0;  // K-blocks filled so far: g / kScB is the batch, g % kScB the entry in it
      bool ok = true;
      auto fill_tile = [&](int t, int64_t kb_lo, int64_t kb_hi) {
        const TileInfo ti = tile_info<kGrouped>(t, args, pref, roff);
        const int64_t a0 = ti.m0 & ~int64_t(3);
        const int64_t rend = ti.m0 + kBM < args.M ? ti.m0 + kBM : args.M;  // rows of this tile: [m0, rend)
        // rows a0 .. rend rounded up to 4 (inside the tensor when M % 4 == 0)
        const uint32_t abytes = static_cast<uint32_t>((rend - a0 + 3) & ~int64_t(3)) * 4u;
        uint32_t sb_bytes = 0;
        if constexpr (kSbGran == 1) {
          // the tail tile of an N that is not a multiple of 256 has 128 columns
          sb_bytes = static_cast<uint32_t>(args.N - ti.n0 < kBN ? args.N - ti.n0 : kBN) * 4u;
        }
        // 128x128-block B scales of the two column halves: lane l holds
        // those of K-blocks sb_kb0 + l and sb_kb0 + 32 + l (reloaded every
        // 64 K-blocks)
        float sbv[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
        int64_t sb_kb0 = kb_lo;
        auto load_sb = [&](int64_t kb0) {
          sb_kb0 = kb0;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int64_t nb = (ti.n0 >> 7) + hh;
            const bool v = nb * 128 < args.N;
            const float* row_p = args.sB + ti.sb_off + nb * KB;
            sbv[hh][0] = v && kb0 + lane < KB ? __ldg(row_p + kb0 + lane) : 0.f;
            sbv[hh][1] = v && kb0 + 32 + lane < KB ? __ldg(row_p + kb0 + 32 + lane) : 0.f;
          }
        };
        if constexpr (kSbGran == 128) load_sb(kb_lo);
        for (int64_t kb = kb_lo; kb < kb_hi; ++kb) {
          const uint32_t bidx = g / kScB, j = g % kScB;
          const uint32_t slot = bidx % kScR;
          const uint32_t sfull = bar_sfull + 8 * slot;
          if (j == 0 && !mbar_wait_warp(bar_sempty + 8 * slot, ((bidx / kScR) & 1u) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* dst = smem + kOffSc + slot * kScSlot + j * kScKb;
          if constexpr (kSbGran == 128) {
            if (kb - sb_kb0 >= 64) load_sb(kb);
            const int d = static_cast<int>(kb - sb_kb0);
            const float b0 = __shfl_sync(0xffffffffu, d < 32 ? sbv[0][0] : sbv[0][1], d & 31);
            const float b1 = __shfl_sync(0xffffffffu, d < 32 ? sbv[1][0] : sbv[1][1], d & 31);
            if (lane < 2) reinterpret_cast<float*>(dst + kScRowBytes)[lane] = lane == 0 ? b0 : b1;
          }
          if (args.sa_bulk) {
            if (elect_one()) {
              mbar_expect_tx(sfull, abytes + sb_bytes);
              bulk_load(smem_u32(dst), args.sA + kb * args.lds_a + a0, abytes, sfull);
              if constexpr (kSbGran == 1)
                bulk_load(smem_u32(dst) + kScRowBytes, args.sB + kb * args.N + ti.n0, sb_bytes, sfull);
            }
          } else {
            float* d4 = reinterpret_cast<float*>(dst);
            for (int r = lane; r < 132; r += 32) {
              const int64_t m = a0 + r;
              d4[r] = m < args.M ? __ldg(args.sA + kb * args.lds_a + m) : 0.f;
            }
            if constexpr (kSbGran == 1) {
              if (elect_one()) {
                mbar_expect_tx(sfull, sb_bytes);
                bulk_load(smem_u32(dst) + kScRowBytes, args.sB + kb * args.N + ti.n0, sb_bytes, sfull);
              }
            }
          }
          __syncwarp();
          ++g;
          if (g % kScB == 0 && elect_one()) mbar_arrive(sfull);  // the batch is complete
          __syncwarp();
        }
      };
      for_each_segment<kStreamK>(args, num_tiles, KB, [&](int t, int64_t lo, int64_t hi) {
        fill_tile(t, lo, hi);
        return ok;
      });
      // close the last batch if it is open (the CTA's last batch may be
      // partial, or a failed wait may have left one half filled)
      if (g % kScB != 0 && elect_one()) mbar_arrive(bar_sfull + 8 * ((g / kScB) % kScR));
      __syncwarp();
      if (!ok && lane == 0 && g > 0) {
        // drain: the copies of the last batches land (bounded) before the
        // CTA exits; the promotion warps consumed every batch otherwise
        const uint32_t last = (g - 1) / kScB;
        for (uint32_t i = 0; i < static_cast<uint32_t>(kScR) && i <= last; ++i) {
          const uint32_t u = last - i;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(bar_sfull + 8 * (u % kScR), (u / kScR) & 1u) && globaltimer_ns() - t0 < 1000000ull) {}
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop, so descriptors and addresses stay
    // warp-uniform; one elected lane issues the MMAs and the commits.
    // (Issued from lane 0 alone, the same loop cost the issuing thread about
    // twice as long per K-block, longer than the K-block's MMAs take.)
    const uint64_t total = cta_kblocks<kStreamK>(args, num_tiles, KB);  // K-blocks of this CTA
    bool ok = true, any = false;
    for (uint64_t g = 0; g < total; ++g) {
      const uint32_t stage = static_cast<uint32_t>(g % kStages);
      const uint32_t phase = static_cast<uint32_t>(g / kStages) & 1u;
      const uint32_t buf = static_cast<uint32_t>(g & 1u);
      const uint32_t bphase = static_cast<uint32_t>(g >> 1) & 1u;
      if (!mbar_wait_warp(bar_tempty + 8 * buf, bphase ^ 1u, abort_flag)) { ok = false; break; }
      if (!mbar_wait_warp(bar_full + 8 * stage, phase, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const uint64_t adesc = smem_desc_k_sw128(sbase + kOffA + stage * kABytes);
      const uint64_t bdesc = smem_desc_k_sw128(sbase + kOffB + stage * kBBytes);
      const uint32_t d = tmem_base + buf * kBN;
      if (elect_one()) {
#pragma unroll
        for (int k = 0; k < kBK / 32; ++k) {
          // K-slice k of the 128-byte swizzled rows: +32 bytes = +2 in the
          // descriptor's 16-byte address units
          mma_f8f6f4(d, adesc + 2u * k, bdesc + 2u * k, kIdesc, k > 0 ? 1u : 0u);
        }
        mma_commit(bar_empty + 8 * stage);
        mma_commit(bar_tfull + 8 * buf);
      }
      __syncwarp();
      any = true;
    }
    if (!ok && any && elect_one()) {
      // drain: wait (bounded) until every MMA issued is done; the commit is
      // made by the elected lane, the one that issued them
      mma_commit(bar_drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bar_drain, 0) && globaltimer_ns() - t0 < 1000000ull) {}
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ promotion
    setmaxnreg_inc<regs_math(kRing)>();
    const int q = warp & 3;         // TMEM lane quadrant this warp may access
    const int h = (warp - 4) >> 2;  // column half of the tile: 0 or 1
    const int row = q * 32 + lane;  // tile-local row
    const uint32_t t_lane = static_cast<uint32_t>(q * 32) << 16;
    uint32_t buf = 0, bphase = 0;
    uint32_t g = 0;  // K-blocks consumed so far: position in the scale ring
    bool ok = true;
    // K-blocks [kb_lo, kb_hi) of tile t: promotion, then the epilogue (whole
    // tile, or the stream-K partial exchange)
    auto tile_work = [&](int t, int64_t kb_lo, int64_t kb_hi) {
      const TileInfo ti = tile_info<kGrouped>(t, args, pref, roff);
      const int64_t m = ti.m0 + row;
      const bool row_ok = m < ti.row_end;
      const int64_t nh = ti.n0 + h * 128;  // first column of this thread's half
      const bool cols_ok = nh < args.N;
      const int a_off = static_cast<int>(ti.m0 & 3);  // the scale slot starts at row m0 rounded down to 4
      float acc[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) acc[j] = 0.f;

      // Scales come either from the scale ring (kRing: a slot entry per
      // K-block, the slot's full barrier waited on at a batch's first entry,
      // a 128x128-block slot released once its last entry is read, a
      // per-column slot only after that K-block's FMAs) or straight from
      // global memory, loaded one K-block ahead (short K: the scales stay in
      // L2 and the load returns within a K-block).
      const float* sb_col = args.sB + ti.sb_off + (nh >> 7) * KB;  // 128x128 scales of this half, by kb
      float sa_next = 0.f, sb_next = 0.f;
      if constexpr (!kRing) {
        sa_next = row_ok ? __ldg(args.sA + kb_lo * args.lds_a + m) : 0.f;
        sb_next = cols_ok ? __ldg(sb_col + kb_lo) : 0.f;
      }

      for (int64_t kb = kb_lo; kb < kb_hi; ++kb) {
        float sa = 0.f, sb = 0.f;
        float sa4[4] = {0.f, 0.f, 0.f, 0.f};  // per-column variant: the scales of this thread's four rows
        const float2* sb2 = nullptr;          // per-column variant: B scales of this half
        if constexpr (kRing) {
          const uint32_t bidx = g / kScB, jb = g % kScB;
          const uint32_t slot = bidx % kScR;
          if (jb == 0 && !mbar_wait_warp(bar_sfull + 8 * slot, (bidx / kScR) & 1u, abort_flag)) { ok = false; break; }
          const uint8_t* ent = smem + kOffSc + slot * kScSlot + jb * kScKb;
          if constexpr (kSbGran == 1) {
            // the 16x256b layout: this thread's rows are q*32 + lane/4 + {0, 8, 16, 24}
            const float* sar = reinterpret_cast<const float*>(ent) + a_off + q * 32 + (lane >> 2);
            sa4[0] = sar[0];
            sa4[1] = sar[8];
            sa4[2] = sar[16];
            sa4[3] = sar[24];
          } else {
            sa = reinterpret_cast<const float*>(ent)[row + a_off];
          }
          if constexpr (kSbGran == 128) {
            sb = reinterpret_cast<const float*>(ent + kScRowBytes)[h];
            if (jb == kScB - 1) {  // the batch's last entry is in registers: the slot is free
              __syncwarp();
              if (lane == 0) mbar_arrive(bar_sempty + 8 * slot);
            }
          } else {
            // columns 8j + 2(lane%4) and +1 of this half, j = 0..15: float2 4j + lane%4
            sb2 = reinterpret_cast<const float2*>(ent + kScRowBytes) + h * 64 + (lane & 3);
          }
        } else {
          sa = sa_next;
          sb = sb_next;
          if (kb + 1 < kb_hi) {
            sa_next = row_ok ? __ldg(args.sA + (kb + 1) * args.lds_a + m) : 0.f;
            sb_next = cols_ok ? __ldg(sb_col + kb + 1) : 0.f;
          }
        }
        if (!mbar_wait_warp(bar_tfull + 8 * buf, bphase, abort_flag)) { ok = false; break; }
        __syncwarp();
        tc_fence_after();
        const uint32_t taddr = tmem_base + t_lane + buf * kBN + h * 128;
        if constexpr (kSbGran == 1) {
          // Per-column B scales: the partial is read in the 16x256b layout,
          // where a thread holds 4 rows x 32 columns (pairs), so it needs 32
          // column scales (16 float2 loads) instead of all 128 of its half.
          // acc[lb*64 + 4j + k]: row q*32 + lb*16 + lane/4 + 8*(k/2), column
          // h*128 + 8j + 2(lane%4) + k%2.
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            uint32_t pa[32], pb[32];
            tmem_ld_16x256b_x8(taddr + ch * 64, pa);
            tmem_ld_16x256b_x8(taddr + (16u << 16) + ch * 64, pb);
            tmem_ld_wait();
            if (ch == 1) {
              // the whole partial of this warp is in registers: free the buffer
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(bar_tempty + 8 * buf);
            }
            // acc += (P * sB) * sA, two columns per packed FP32 instruction
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              float* a0 = acc + 4 * (ch * 8 + j);
              float* a1 = a0 + 64;
              const float2 bj = sb2[4 * (ch * 8 + j)];
              float t0, t1, t2, t3;
              mul2(t0, t1, __uint_as_float(pa[4 * j + 0]), __uint_as_float(pa[4 * j + 1]), bj.x, bj.y);
              mul2(t2, t3, __uint_as_float(pa[4 * j + 2]), __uint_as_float(pa[4 * j + 3]), bj.x, bj.y);
              fma2(a0[0], a0[1], t0, t1, sa4[0], sa4[0]);
              fma2(a0[2], a0[3], t2, t3, sa4[1], sa4[1]);
              mul2(t0, t1, __uint_as_float(pb[4 * j + 0]), __uint_as_float(pb[4 * j + 1]), bj.x, bj.y);
              mul2(t2, t3, __uint_as_float(pb[4 * j + 2]), __uint_as_float(pb[4 * j + 3]), bj.x, bj.y);
              fma2(a1[0], a1[1], t0, t1, sa4[2], sa4[2]);
              fma2(a1[2], a1[3], t2, t3, sa4[3], sa4[3]);
            }
          }
        } else {
          const float scale = sa * sb;
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            uint32_t p[64];
            tmem_ld_32x32b_x64(taddr + c2 * 64, p);
            tmem_ld_wait();
            if (c2 == 1) {
              // the whole partial of this warp is in registers: free the buffer
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(bar_tempty + 8 * buf);
            }
            // acc += P * scale, two columns per packed FP32 instruction
#pragma unroll
            for (int j = 0; j < 64; j += 2)
              fma2(acc[c2 * 64 + j], acc[c2 * 64 + j + 1], __uint_as_float(p[j]), __uint_as_float(p[j + 1]), scale,
                   scale);
          }
        }
        if constexpr (kSbGran == 1) {
          if (g % kScB == kScB - 1) {  // this K-block was its slot's last: the slot is free
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_sempty + 8 * ((g / kScB) % kScR));
          }
        }
        ++g;
        buf ^= 1u;
        if (buf == 0) bphase ^= 1u;
      }
      if constexpr (kStreamK) {
        // the exchange below synchronizes the promotion warps: they all
        // leave together if any of them gave up a wait
        if (promo_bar_or(!ok)) {
          ok = false;
          return;
        }
        if (kb_lo > 0) {
          // this CTA holds the later K-blocks of a split tile: leave the FP32
          // partial in its workspace slot and raise its flag
          float4* dst = args.ws + (static_cast<size_t>(blockIdx.x) * 2 + h) * 32 * 128 + row;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            dst[j * 128] = make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
          __threadfence();
          promo_bar_sync();
          if (warp == 4 && lane == 0) st_release_gpu(args.flags + blockIdx.x, args.epoch);
          return;
        }
        if (kb_hi < KB) {
          // this CTA holds the first K-blocks of a split tile: add the
          // partials of the CTAs holding the rest, in CTA order
          const int64_t all = static_cast<int64_t>(num_tiles - args.sk_tile0) * KB;
          const int64_t tile_end = static_cast<int64_t>(t - args.sk_tile0 + 1) * KB;
          for (int64_t j = static_cast<int64_t>(blockIdx.x) + 1; j < gridDim.x; ++j) {
            const int64_t bj = streamk_begin(all, j, gridDim.x);
            if (bj >= tile_end) break;
            if (streamk_begin(all, j + 1, gridDim.x) == bj) continue;  // CTA j has no K-blocks
            if (warp == 4 && lane == 0) {
              const uint64_t t0 = globaltimer_ns();
              while (ld_acquire_gpu(args.flags + j) != args.epoch) {
                if (*abort_flag) break;
                if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
                  atomicCAS(&g_status_word, 0u, kStatusTimeout);
                  *abort_flag = 1;
                  break;
                }
                __nanosleep(64);
              }
            }
            promo_bar_sync();
            const float4* src = args.ws + (static_cast<size_t>(j) * 2 + h) * 32 * 128 + row;
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              const float4 v = __ldcg(src + jj * 128);
              acc[4 * jj + 0] += v.x;
              acc[4 * jj + 1] += v.y;
              acc[4 * jj + 2] += v.z;
              acc[4 * jj + 3] += v.w;
            }
            promo_bar_sync();  // every thread has read slot j: its flag may drop
            if (warp == 4 && lane == 0) args.flags[j] = 0u;
          }
        }
      } else {
        if (!ok) return;
      }

      // ---- epilogue: this warp's 32 rows x 128 columns ----
      // Whole-warp row blocks go out through shared memory and TMA stores in
      // 32-row x 32-byte chunks (two chunk buffers per warp, so the write of
      // one chunk overlaps the store of the previous); TMA clips rows past
      // the end of C.  A grouped tile whose expert ends inside this warp's
      // rows (the next expert's rows follow) stores its valid rows directly.
      const int64_t wrow0 = ti.m0 + q * 32;
      const bool via_tma = ti.row_end >= args.M || wrow0 + 32 <= ti.row_end;
      if (cols_ok && wrow0 < ti.row_end) {
        if (via_tma) {
          uint8_t* stg = smem + kOffStage + (warp - 4) * 2 * kChunkBytes;
          constexpr int kCols = kOutF32 ? 8 : 16;  // columns per 32-byte chunk row
#pragma unroll
          for (int c = 0; c < 128 / kCols; ++c) {
            uint8_t* cb = stg + (c & 1) * kChunkBytes;
            if (lane == 0) bulk_wait_read<1>();  // the chunk buffer's previous store has read it
            __syncwarp();
            if constexpr (kSbGran == 1) {
              // the 16x256b layout (see the promotion): rows lb*16 + lane/4
              // + 8*hi of the warp's 32, column pairs 2(lane%4) of each
              // 8-column block
#pragma unroll
              for (int lb = 0; lb < 2; ++lb) {
#pragma unroll
                for (int hi = 0; hi < 2; ++hi) {
                  uint8_t* rp = cb + (lb * 16 + (lane >> 2) + 8 * hi) * 32;
                  const float* a = acc + lb * 64 + 2 * hi;
                  if constexpr (kOutF32) {
                    *reinterpret_cast<uint2*>(rp + 8 * (lane & 3)) =
                        make_uint2(__float_as_uint(a[4 * c]), __float_as_uint(a[4 * c + 1]));
                  } else {
                    *reinterpret_cast<uint32_t*>(rp + 4 * (lane & 3)) = cvt_bf16x2(a[8 * c], a[8 * c + 1]);
                    *reinterpret_cast<uint32_t*>(rp + 16 + 4 * (lane & 3)) = cvt_bf16x2(a[8 * c + 4], a[8 * c + 5]);
                  }
                }
              }
            } else {
            uint4 v0, v1;
            if constexpr (kOutF32) {
              v0 = make_uint4(__float_as_uint(acc[8 * c + 0]), __float_as_uint(acc[8 * c + 1]),
                              __float_as_uint(acc[8 * c + 2]), __float_as_uint(acc[8 * c + 3]));
              v1 = make_uint4(__float_as_uint(acc[8 * c + 4]), __float_as_uint(acc[8 * c + 5]),
                              __float_as_uint(acc[8 * c + 6]), __float_as_uint(acc[8 * c + 7]));
            } else {
              v0 = make_uint4(cvt_bf16x2(acc[16 * c + 0], acc[16 * c + 1]), cvt_bf16x2(acc[16 * c + 2], acc[16 * c + 3]),
                              cvt_bf16x2(acc[16 * c + 4], acc[16 * c + 5]), cvt_bf16x2(acc[16 * c + 6], acc[16 * c + 7]));
              v1 = make_uint4(cvt_bf16x2(acc[16 * c + 8], acc[16 * c + 9]),
                              cvt_bf16x2(acc[16 * c + 10], acc[16 * c + 11]),
                              cvt_bf16x2(acc[16 * c + 12], acc[16 * c + 13]),
                              cvt_bf16x2(acc[16 * c + 14], acc[16 * c + 15]));
            }
            *reinterpret_cast<uint4*>(cb + lane * 32) = v0;
            *reinterpret_cast<uint4*>(cb + lane * 32 + 16) = v1;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmC, smem_u32(cb), static_cast<int32_t>(nh + c * kCols), static_cast<int32_t>(wrow0));
              bulk_commit();
            }
          }
        } else if (kSbGran != 1 && row_ok) {  // (dense per-column tiles always go through TMA)
          if constexpr (kOutF32) {
            float4* out = reinterpret_cast<float4*>(static_cast<float*>(args.C) + m * args.N + nh);
#pragma unroll
            for (int j = 0; j < 32; ++j)
              out[j] = make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
          } else {
            uint4* out = reinterpret_cast<uint4*>(static_cast<uint16_t*>(args.C) + m * args.N + nh);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              out[j] = make_uint4(cvt_bf16x2(acc[8 * j + 0], acc[8 * j + 1]), cvt_bf16x2(acc[8 * j + 2], acc[8 * j + 3]),
                                  cvt_bf16x2(acc[8 * j + 4], acc[8 * j + 5]), cvt_bf16x2(acc[8 * j + 6], acc[8 * j + 7]));
          }
        }
      }
    };
    for_each_segment<kStreamK>(args, num_tiles, KB, [&](int t, int64_t lo, int64_t hi) {
      tile_work(t, lo, hi);
      return ok;
    });
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
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace fp8q
