// chain_kernel.cuh -- the persistent fused-chain kernel for sm_103a.
//
// One CTA per SM loops over 128-row output tiles (BOLT notes, "Persistent kernel
// (GEMM/Conv) fusion").  The CTA owns every N0 and N1 column of its rows ("Threadblock
// residence": ThreadBlock_N = GEMM_N), so GEMM1 never needs another block's data:
//
//   warp 0      TMA producer: A (or one conv tap of x) and weight K-chunks -> smem ring
//   warp 1      TMEM allocator and tcgen05.mma issuer (GEMM0 into TMEM, GEMM1 from P)
//   (both run as converged warps; one elected lane issues each TMA / MMA / commit)
//   warps 2..9  epilogue, two warpgroups: TMEM -> registers -> act -> fp16/bf16 ->
//               (chain) P tile in shared memory, the operand of GEMM1
//               ("Shared-memory-resident fusion": the accumulator tile is staged in
//               shared memory and read back by the second GEMM, Figure 7)
//               (last stage) output tile in shared memory -> TMA store to global
//
// Modes
//   MODE_CHAIN   GEMM0 -> epi0 -> P -> GEMM1 -> epi1 -> global
//   MODE_SINGLE  GEMM0 -> epi0 -> global             (one operator of the unfused path)
//   MODE_POOL    conv GEMM -> 2x2 max -> ReLU -> global (Welder notes, Figure 5:
//                the (2,2,F) reuse tile is reduced in registers and never leaves the chip)
//   MODE_CHAIN3  GEMM0 -> epi0 -> P0 -> GEMM1 -> epi1 -> P1 -> GEMM2 -> epi2 -> global
//                (BOLT notes, "Enabling deeper operator fusion": more than two GEMMs in
//                one persistent kernel); weights resident, two tiles in flight
//
// A operand
//   2-D: rows of A[M, K0] in 128 x 64 boxes.
//   4-D (implicit GEMM, interview notes "Conv optimisation", item 2): for tap (r, s) and
//   channel block cb, one box x[n, ho0+r-pad .. +8, wo0+s-pad .. +16, cb*64 .. +64] of
//   an 8 x 16 output-pixel tile; coordinates outside the image read as zero, which is the
//   conv's zero padding.  The box lands in shared memory as 128 rows x 128 B, exactly the
//   K-major 128B-swizzled layout tcgen05 reads, so no im2col buffer exists anywhere.
//
// Bias: each GEMM's last MMA adds the bias to its accumulator (D += ONES . BIAS, see
// fill_bias_operands), so epilogues apply only the activation and the rounding.
//
// Two tiles in flight: when TMEM and shared memory allow (acc_dual), tile i uses
// accumulator / P / staging buffer i & 1 and the two epilogue warpgroups take alternate
// tiles, so GEMM0 of tile i+2 and GEMM1 of tile i+1 run while the epilogue of tile i
// drains.  The MMA issue order is G0(0), G0(1), then G1(j), G0(j+2) for j = 0, 1, ...
// Otherwise (one buffer) it is G0(0), then G1(j), G0(j+1), and both warpgroups split the
// columns of every tile.  With P kept in TMEM (N0 > 128) tiles run in pairs: G0(k),
// G0(k+1), G1(k), G1(k+1), each tile's P packed in place over its GEMM0 columns.  Wide
// chains (256 < N0 <= 512, the WIDE instantiation) run GEMM0 in two passes over the
// halves of N0, each warpgroup packing one half's P while the other pass or GEMM1 runs;
// D1 sits in the half computed first, which alternates from tile to tile.  The schedules
// are separate instantiations (WIDE, PAIR, NOPAIR) so that each kernel carries only its
// own loops, and every unit is compiled once without the event trace and once with it.
//
// Every wait is bounded (see ptx.cuh); on a timeout all roles leave their loops, the MMA
// issuer drains its MMAs, the producer drains its copies, and TMEM is freed.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernel_params.h"
#include "ptx.cuh"

// Every kernel unit is compiled twice: without the event trace (B2B_TRACE 0, the kernels
// every launch uses) and with it (B2B_TRACE 1, launched only while a trace buffer is set).
// The two builds live in the namespaces b2b::plain and b2b::traced.
#ifndef B2B_TRACE
#define B2B_TRACE 0
#endif
#if B2B_TRACE
#define B2B_KNS traced
#else
#define B2B_KNS plain
#endif

namespace b2b {
namespace B2B_KNS {

// Barrier slots (8 bytes each) at p.off_bar.
enum : uint32_t {
  BAR_FULL0 = 0,
  BAR_EMPTY0 = kMaxStages,
  BAR_WFULL = 2 * kMaxStages,
  BAR_ACC_FULL0 = BAR_WFULL + 1,
  BAR_ACC_EMPTY0 = BAR_ACC_FULL0 + kMaxBufs,
  BAR_P_FULL0 = BAR_ACC_EMPTY0 + kMaxBufs,
  BAR_D1_FULL0 = BAR_P_FULL0 + kMaxBufs,
  BAR_P1_FULL0 = BAR_D1_FULL0 + kMaxBufs,   // three-operator chain: P1 published
  BAR_D2_FULL0 = BAR_P1_FULL0 + kMaxBufs,   // three-operator chain: GEMM2 accumulator ready
  BAR_MMA_DONE = BAR_D2_FULL0 + kMaxBufs,
  BAR_BIAS_READY = BAR_MMA_DONE + 1,
  BAR_W0C0 = BAR_BIAS_READY + 1,            // resident W0 beside streamed W1: one per K chunk
  BAR_COUNT = BAR_W0C0 + kMaxW0Chunks,
};
constexpr uint32_t kBarRegionBytes = 512;   // barriers, then TMEM slot and abort flag
static_assert(8u * BAR_COUNT + 8u <= kBarRegionBytes, "barrier region too small");

struct TileCoord {
  int32_t m0;              // 2-D: first row
  int32_t n, ho0, wo0;     // 4-D: image, first output row, first output column
};

template <bool A4D>
__device__ __forceinline__ TileCoord tile_coord(const ChainParams& p, int32_t t) {
  TileCoord c{0, 0, 0, 0};
  if constexpr (A4D) {
    const int32_t per_img = p.tiles_h * p.tiles_w;
    c.n = t / per_img;
    const int32_t rem = t - c.n * per_img;
    const int32_t th = rem / p.tiles_w;
    c.ho0 = th * 8;
    c.wo0 = (rem - th * p.tiles_w) * 16;
  } else {
    c.m0 = t * kBlockM;
  }
  return c;
}

// Optional event trace of one CTA.  The buffer holds four regions of trace_cap / 4 events,
// one per role (producer, MMA issuer, epilogue group 0, group 1); each role appends to its
// own region with plain stores, so tracing costs a few instructions per event.  An event
// is two words: %globaltimer (ns; one clock for all warps and SMs), and
// code | group << 8 | tile index << 16 | 1 << 63.
// Without B2B_TRACE the tracer is empty: even a disabled trace (a pointer test per event)
// cost the FFN chain 5 % and the 1x1 conv chain 8 % per launch.
#if B2B_TRACE
struct Tracer {
  unsigned long long* base = nullptr;
  uint32_t n = 0, cap = 0;
  __device__ __forceinline__ Tracer(const ChainParams& p, uint32_t region, uint32_t leader,
                                    uint32_t first = 0) {
    if (p.trace != nullptr && blockIdx.x == p.trace_cta && leader != 0u) {
      cap = p.trace_cap / 4u;
      base = p.trace + 2ull * cap * region;
      n = first;
    }
  }
  __device__ __forceinline__ void operator()(uint32_t code, uint32_t group, int it) {
    if (base == nullptr || n >= cap) return;
    base[2 * n] = static_cast<unsigned long long>(global_timer_ns());
    base[2 * n + 1] = code | (group << 8) | (static_cast<unsigned long long>(it) << 16) |
                      (1ull << 63);
    ++n;
  }
};
#else
struct Tracer {
  __device__ __forceinline__ Tracer(const ChainParams&, uint32_t, uint32_t, uint32_t = 0) {}
  __device__ __forceinline__ void operator()(uint32_t, uint32_t, int) {}
};
#endif

// Number of tiles this CTA processes (tiles blockIdx.x, blockIdx.x + gridDim.x, ...).
__device__ __forceinline__ int local_tiles(const ChainParams& p) {
  const int b = static_cast<int>(blockIdx.x), g = static_cast<int>(gridDim.x);
  return b < p.num_tiles ? (p.num_tiles - 1 - b) / g + 1 : 0;
}

// A walker over the ring slots [start, end): the slot and phase parity of successive
// stages, stepped by one per stage.  (No division per stage: with N = 64 the MMA issuers'
// pauses between ring stages are what bounds a launch, and a slot computed from the tile
// and stage index with two integer divisions made the conv + pool kernel ~10 % slower.)
struct SubRing {
  int start, end, slot;
  uint32_t phase;
};
__device__ __forceinline__ SubRing make_subring(int start, int end) {
  SubRing r;
  r.start = start;
  r.end = end;
  r.slot = start;
  r.phase = 0u;
  return r;
}
__device__ __forceinline__ void advance_subring(SubRing& r) {
  if (++r.slot == r.end) {
    r.slot = r.start;
    r.phase ^= 1u;
  }
}

// Two MMA issuers (two_issuers(MODE, TWO)): each takes the tiles of one parity and the
// ring is split into two sub-rings, [0, S/2) for even tiles and [S/2, S) for odd ones, so
// that each sub-ring has one consumer that takes its slots in order (a consumer further
// ahead than one phase of a slot would alias the barrier's phase parity).  The tiles of one
// parity take consecutive positions in their sub-ring.
__device__ __forceinline__ SubRing subring_of(const ChainParams& p, int parity) {
  const int s0 = static_cast<int>(p.num_stages) >> 1;
  return parity ? make_subring(s0, static_cast<int>(p.num_stages)) : make_subring(0, s0);
}

// Buffer of the CTA's it-th tile and the phase parity of its barriers.
__device__ __forceinline__ uint32_t buf_of(const ChainParams& p, int it) {
  return static_cast<uint32_t>(it) & ((1u << p.nbuf_log2) - 1u);
}
__device__ __forceinline__ uint32_t use_of(const ChainParams& p, int it) {
  return (static_cast<uint32_t>(it) >> p.nbuf_log2) & 1u;
}

// Bounded wait executed by a whole warp; the lanes agree on the outcome.
__device__ __forceinline__ bool warp_mbar_wait(uint32_t bar, uint32_t parity,
                                               const ChainParams& p,
                                               volatile uint32_t* abort_flag, uint32_t site,
                                               int32_t t) {
  const bool ok =
      mbar_wait(bar, parity, p.wait_limit_ns, abort_flag, p.err, p.kernel_id, site, t);
  return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------------------------------------------
// producer (one warp; the elected lane issues)
// ------------------------------------------------------------------------------------
// Position of a GEMM0 K chunk: filter tap (r, s), its index t = r * S + s, and the
// channel block cb within the tap (2-D A: t = r = s = 0 and cb = chunk index).  Advanced
// with counters so that the issue loops do no division.
struct KPos {
  int r = 0, s = 0, t = 0, cb = 0;
  __device__ __forceinline__ void next(const ChainParams& p) {
    if (++cb == p.kc_per_tap) {
      cb = 0;
      ++t;
      if (++s == p.S) { s = 0; ++r; }
    }
  }
  // Halo stages: channel block fastest, then the column tap s (all row taps at once).
  __device__ __forceinline__ void next_halo(const ChainParams& p) {
    if (++cb == p.kc_per_tap) { cb = 0; ++s; }
  }
};

template <int MODE, bool A4D, bool W0MN, bool W1MN>
__device__ __forceinline__ void load_a_chunk(uint32_t lead, const ChainParams& p,
                                             const CUtensorMap* tmA, uint32_t dst,
                                             const TileCoord& tc, const KPos& k, uint32_t bar,
                                             uint64_t pol) {
  if constexpr (A4D) {
    // output pixel (ho, wo) reads input (stride * ho + r - pad, stride * wo + s - pad); the
    // map's element strides make the box take every stride-th pixel
    tma_load_4d(lead, dst, tmA, bar, k.cb * kChunkK, tc.wo0 * p.stride + k.s - p.pad,
                tc.ho0 * p.stride + k.r - p.pad, tc.n, pol);
  } else {
    tma_load_2d(lead, dst, tmA, bar, k.cb * kChunkK, tc.m0, pol);
  }
}

template <bool A4D, bool W0MN>
__device__ __forceinline__ void load_w0_chunk(uint32_t lead, const ChainParams& p,
                                              const CUtensorMap* tmW0, uint32_t dst,
                                              const KPos& k, uint32_t bar, uint64_t pol) {
  if constexpr (W0MN) {
    // W0[K0][N0] row-major: a 64 (N) x 64 (K) box per 64-wide N block, 8 KiB apart; with
    // the [N0/64][K0][64] view, all blocks in one box.
    if (p.w0_box3) {
      tma_load_3d(lead, dst, tmW0, bar, 0, k.cb * kChunkK, 0, pol);
      return;
    }
    const int nblk = (p.N0p + 63) >> 6;
    for (int nb = 0; nb < nblk; ++nb)
      tma_load_2d(lead, dst + nb * 8192u, tmW0, bar, nb * 64, k.cb * kChunkK, pol);
  } else if constexpr (A4D) {
    // W0[C0][R*S][C]: the 64-channel block cb of tap t for all C0 rows.
    tma_load_3d(lead, dst, tmW0, bar, k.cb * kChunkK, k.t, 0, pol);
  } else {
    tma_load_2d(lead, dst, tmW0, bar, k.cb * kChunkK, 0, pol);
  }
}

// Wide chains: the K chunk's 64-wide N blocks [4h, 4h + 4) of W0 (half h of N0): one box
// of four blocks in the [N0/64][K0][64] view (blocks past N0 zero-filled), else one 2-D box
// per block.  Returns the bytes the loads deliver.
__device__ __forceinline__ uint32_t w0_half_bytes(const ChainParams& p, int h) {
  if (h == 0 || p.w0_box3) return p.w0_chunk_bytes;
  return static_cast<uint32_t>(((p.N0p + 63) >> 6) - 4) * 8192u;
}
__device__ __forceinline__ void load_w0_half(uint32_t lead, const ChainParams& p,
                                             const CUtensorMap* tmW0, uint32_t dst, int kc,
                                             int h, uint32_t bar, uint64_t pol) {
  if (p.w0_box3) {
    tma_load_3d(lead, dst, tmW0, bar, 0, kc * kChunkK, 4 * h, pol);
    return;
  }
  const int nblk = min((p.N0p + 63) >> 6, 4 * h + 4);
  for (int nb = 4 * h; nb < nblk; ++nb)
    tma_load_2d(lead, dst + (nb - 4 * h) * 8192u, tmW0, bar, nb * 64, kc * kChunkK, pol);
}

template <bool W1MN>
__device__ __forceinline__ void load_w1_chunk(uint32_t lead, const ChainParams& p,
                                              const CUtensorMap* tmW1, uint32_t dst, int kc1,
                                              uint32_t bar, uint64_t pol) {
  if constexpr (W1MN) {
    if (p.w1_box3) {
      tma_load_3d(lead, dst, tmW1, bar, 0, kc1 * kChunkK, 0, pol);
      return;
    }
    const int nblk = (p.N1p + 63) >> 6;
    for (int nb = 0; nb < nblk; ++nb)
      tma_load_2d(lead, dst + nb * 8192u, tmW1, bar, nb * 64, kc1 * kChunkK, pol);
  } else {
    tma_load_2d(lead, dst, tmW1, bar, kc1 * kChunkK, 0, pol);
  }
}

// L2 prefetch of tile t's rows of a 2-D A (contiguous, row-major).  Prefetches only warm
// L2, so they may run before the previous kernel's writes are visible: L2 is where those
// writes land.  The implicit-GEMM conv A has no per-tile contiguous range and is skipped.
__device__ __forceinline__ void prefetch_a_tile(const ChainParams& p, int32_t t) {
  if (p.pf_a == nullptr || t >= p.num_tiles) return;
  const uint64_t off = static_cast<uint64_t>(t) * p.pf_a_tile_bytes;
  const uint64_t n = min(static_cast<uint64_t>(p.pf_a_tile_bytes), p.pf_a_bytes - off);
  bulk_prefetch_l2(p.pf_a + off, static_cast<uint32_t>(n));
}

template <int MODE, bool A4D, bool W0MN, bool W1MN, bool WIDE, bool PAIR, bool NOPAIR, bool W0RES,
          bool TWO>
__device__ void producer_role(const ChainParams& p, const CUtensorMap* tmA,
                              const CUtensorMap* tmW0, const CUtensorMap* tmW1, uint32_t base,
                              uint32_t bars, volatile uint32_t* abort_flag) {
  // Tile-pair instantiations are launched with streamed weights only, or (W0RES) with W0
  // alone resident: then the ring carries A chunks and W1 chunks.
  const bool resident = !PAIR && p.resident != 0;
  const bool stream_w0 = !resident && !W0RES;
  const uint32_t lead = elect_one();
  const uint64_t pol_stream = l2_policy_evict_first();
  const uint64_t pol_keep = l2_policy_evict_last();
  Tracer trace(p, 0, lead);
  grid_dependency_wait();   // global memory only after the previous grid has completed
  trace(EV_PROD_START, 0, 0);
  uint32_t issued = 0, issued_parity = 0;   // per-stage: a fill in flight, and its parity
  bool w_issued = false;
  uint32_t w0_issued = 0;                   // W0RES: resident W0 chunks requested
  bool ok = true;

  if (resident) {
    const uint32_t wbar = bars + 8u * BAR_WFULL;
    uint32_t total = p.kchunks0 * p.w0_chunk_bytes;
    if (MODE == MODE_CHAIN || MODE == MODE_CHAIN3) total += p.kchunks1 * p.w1_chunk_bytes;
    mbar_arrive_expect_tx_if(lead, wbar, total);
    KPos k;
    for (int kc = 0; kc < p.kchunks0; ++kc, k.next(p))
      load_w0_chunk<A4D, W0MN>(lead, p, tmW0, base + p.off_w0 + kc * p.w0_chunk_bytes, k, wbar,
                               pol_keep);
    if (MODE == MODE_CHAIN || MODE == MODE_CHAIN3)
      for (int kc1 = 0; kc1 < p.kchunks1; ++kc1)
        load_w1_chunk<W1MN>(lead, p, tmW1, base + p.off_w1 + kc1 * p.w1_chunk_bytes, kc1, wbar,
                            pol_keep);
    w_issued = true;
  }

  int stage = 0;
  uint32_t phase = 0;
  // two issuers: the sub-rings of the next tile to load (its parity) and of the one after
  const bool two = two_issuers(MODE, TWO) && p.two_issuers != 0;
  SubRing sr_cur = subring_of(p, 0), sr_next = subring_of(p, 1);
  auto acquire = [&](int32_t t) -> bool {   // waits until ring slot `stage` is free
    return warp_mbar_wait(bars + 8u * (BAR_EMPTY0 + stage), phase ^ 1u, p, abort_flag,
                          SITE_PRODUCER_EMPTY, t);
  };
  auto advance = [&]() {
    issued |= 1u << stage;
    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
    if (++stage == static_cast<int>(p.num_stages)) { stage = 0; phase ^= 1u; }
  };
  // A (and streamed W0) chunks of the it-th tile of this CTA.
  auto load_g0 = [&](int it) -> bool {
    const int32_t t = blockIdx.x + it * gridDim.x;
    const TileCoord tc = tile_coord<A4D>(p, t);
    KPos k;
    for (int kc = 0; kc < p.kstages0; ++kc) {
      if (two) {   // (tiles are loaded in order: it's parity is sr_cur's)
        stage = sr_cur.slot;
        phase = sr_cur.phase;
        advance_subring(sr_cur);
      }
      if (W0RES && it == 0) {
        // The resident W0, chunk by chunk beside the CTA's first tile, so that its first
        // MMAs wait for one chunk, not for the whole matrix.
        const uint32_t wb = bars + 8u * (BAR_W0C0 + kc);
        mbar_arrive_expect_tx_if(lead, wb, p.w0_chunk_bytes);
        load_w0_chunk<A4D, W0MN>(lead, p, tmW0, base + p.off_w0 + kc * p.w0_chunk_bytes, k, wb,
                                 pol_keep);
        w0_issued |= 1u << kc;
      }
      if (!acquire(t)) return false;
      trace(EV_PROD_ACQUIRE, kc, it);
      const uint32_t fb = bars + 8u * (BAR_FULL0 + stage);
      const uint32_t sbase = base + p.off_ring + stage * p.stage_bytes;
      mbar_arrive_expect_tx_if(lead, fb, p.a_stage_bytes + (stream_w0 ? p.w0_chunk_bytes : 0u));
      load_a_chunk<MODE, A4D, W0MN, W1MN>(lead, p, tmA, sbase, tc, k, fb, pol_stream);
      if (stream_w0)
        load_w0_chunk<A4D, W0MN>(lead, p, tmW0, sbase + kABytes, k, fb, pol_keep);
      if (A4D && p.halo) k.next_halo(p); else k.next(p);
      // (Tile 0's A, and tile 1's when the CTA has more tiles, were prefetched into L2 at
      // the start.  Prefetching tile it + 2 here as well measured 0-1.5 % slower on every
      // workload: the ring's own loads keep HBM as busy.)
      trace(EV_PROD_ISSUED, kc, it);
      advance();
    }
    if (two) {
      const SubRing x = sr_cur;
      sr_cur = sr_next;
      sr_next = x;
    }
    return true;
  };
  // Streamed W1 for GEMM1 of the it-th tile (or, with w1_group, of the pair it, it + 1):
  // w1_per_stage chunks per ring stage.
  auto load_g1 = [&](int it) -> bool {
    if (MODE != MODE_CHAIN || resident) return true;
    const int32_t t = blockIdx.x + it * gridDim.x;
    for (int kc1 = 0; kc1 < p.kchunks1;) {
      if (!acquire(t)) return false;
      const int n = min(static_cast<int>(p.w1_per_stage), p.kchunks1 - kc1);
      const uint32_t fb = bars + 8u * (BAR_FULL0 + stage);
      const uint32_t sbase = base + p.off_ring + stage * p.stage_bytes;
      mbar_arrive_expect_tx_if(lead, fb, static_cast<uint32_t>(n) * p.w1_chunk_bytes);
      for (int j = 0; j < n; ++j)
        load_w1_chunk<W1MN>(lead, p, tmW1, sbase + j * p.w1_chunk_bytes, kc1 + j, fb, pol_keep);
      trace(EV_PROD_W1_ISSUED, kc1, it);
      advance();
      kc1 += n;
    }
    return true;
  };

  // Wide chains, tile it, half h of N0: GEMM0's A chunks with that half's W0 chunks, and
  // W1's rows of that half (w1_per_stage chunks per ring stage).
  auto load_g0_half = [&](int it, int h) -> bool {
    const int32_t t = blockIdx.x + it * gridDim.x;
    const TileCoord tc = tile_coord<A4D>(p, t);
    const uint32_t wbytes = w0_half_bytes(p, h);
    KPos k;
    for (int kc = 0; kc < p.kchunks0; ++kc, k.next(p)) {
      if (!acquire(t)) return false;
      trace(EV_PROD_ACQUIRE, kc, it);
      const uint32_t fb = bars + 8u * (BAR_FULL0 + stage);
      const uint32_t sbase = base + p.off_ring + stage * p.stage_bytes;
      mbar_arrive_expect_tx_if(lead, fb, kABytes + wbytes);
      load_a_chunk<MODE, A4D, W0MN, W1MN>(lead, p, tmA, sbase, tc, k, fb, pol_stream);
      load_w0_half(lead, p, tmW0, sbase + kABytes, kc, h, fb, pol_keep);
      trace(EV_PROD_ISSUED, kc, it);
      advance();
    }
    return true;
  };
  auto load_w1_half = [&](int it, int h) -> bool {
    const int32_t t = blockIdx.x + it * gridDim.x;
    const int first = 4 * h, end = h == 0 ? min(4, p.kchunks1) : p.kchunks1;
    for (int kc1 = first; kc1 < end;) {
      if (!acquire(t)) return false;
      const int n = min(static_cast<int>(p.w1_per_stage), end - kc1);
      const uint32_t fb = bars + 8u * (BAR_FULL0 + stage);
      const uint32_t sbase = base + p.off_ring + stage * p.stage_bytes;
      mbar_arrive_expect_tx_if(lead, fb, static_cast<uint32_t>(n) * p.w1_chunk_bytes);
      for (int j = 0; j < n; ++j)
        load_w1_chunk<W1MN>(lead, p, tmW1, sbase + j * p.w1_chunk_bytes, kc1 + j, fb, pol_keep);
      trace(EV_PROD_W1_ISSUED, kc1, it);
      advance();
      kc1 += n;
    }
    return true;
  };

  const int ntiles = local_tiles(p);
  if constexpr (MODE == MODE_CHAIN && WIDE) {
    // As the MMA issuer consumes: per tile, GEMM0 over the first half of N0 (the lower on
    // even tiles, the upper on odd ones), then over the other half, then W1 in that order.
    for (int it = 0; ok && it < ntiles; ++it) {
      const int f = it & 1;
      ok = load_g0_half(it, f);
      if (ok) ok = load_g0_half(it, f ^ 1);
      if (ok) ok = load_w1_half(it, f);
      if (ok) ok = load_w1_half(it, f ^ 1);
    }
  } else if (MODE == MODE_CHAIN && (PAIR || (!NOPAIR && p.p_tmem))) {
    // Pairs: G0(0), G0(1), then G1(k), G1(k+1), G0(k+2), G0(k+3) -- as the MMA issuer.
    for (int it = 0; ok && it < 2 && it < ntiles; ++it) ok = load_g0(it);
    for (int k = 0; ok && k < ntiles; k += 2) {
      if (p.w1_group) {
        ok = load_g1(k);
      } else {
        ok = load_g1(k);
        if (ok && k + 1 < ntiles) ok = load_g1(k + 1);
      }
      if (ok && k + 2 < ntiles) ok = load_g0(k + 2);
      if (ok && k + 3 < ntiles) ok = load_g0(k + 3);
    }
  } else if (MODE == MODE_CHAIN) {
    // Same order as the MMA issuer consumes: G0(0..L-1), then G1(j), G0(j+L).
    const int L = 1 << p.nbuf_log2;
    for (int it = 0; ok && it < L && it < ntiles; ++it) ok = load_g0(it);
    for (int j = 0; ok && j < ntiles; ++j) {
      ok = load_g1(j);
      if (ok && j + L < ntiles) ok = load_g0(j + L);
    }
  } else {
    for (int it = 0; ok && it < ntiles; ++it) ok = load_g0(it);
  }

  if (!ok) {
    // Gave up: let the copies this thread started land before the CTA can exit.
    const uint64_t drain_ns = 100000000ull;
    for (uint32_t s = 0; s < p.num_stages; ++s)
      if (issued & (1u << s))
        (void)mbar_wait(bars + 8u * (BAR_FULL0 + s), (issued_parity >> s) & 1u, drain_ns,
                        nullptr, p.err, p.kernel_id, SITE_PRODUCER_DRAIN, 0);
    if (w_issued)
      (void)mbar_wait(bars + 8u * BAR_WFULL, 0u, drain_ns, nullptr, p.err, p.kernel_id,
                      SITE_PRODUCER_DRAIN, 0);
    for (uint32_t c = 0; c < static_cast<uint32_t>(kMaxW0Chunks); ++c)
      if (w0_issued & (1u << c))
        (void)mbar_wait(bars + 8u * (BAR_W0C0 + c), 0u, drain_ns, nullptr, p.err, p.kernel_id,
                        SITE_PRODUCER_DRAIN, 0);
  }
}

// ------------------------------------------------------------------------------------
// MMA issuer (one thread)
// ------------------------------------------------------------------------------------
// Issues the MMAs of one 64-wide K chunk: D (+)= A . B over `nks` 16-wide K steps (the
// first chunk of a GEMM overwrites D; the bias is added by the GEMM's last MMA).  The
// descriptors of consecutive K steps differ only in their start-address field (32 B per
// step for K-major operands, 2 KiB for an MN-major one), so each step is one add; with
// small N the single issuing thread is otherwise the bottleneck.
template <bool BMN>
__device__ __forceinline__ void issue_chunk(uint32_t lead, uint32_t d, uint64_t adesc,
                                            uint64_t bdesc, uint32_t idesc, int nks, bool first) {
  constexpr uint64_t kAStep = 32u >> 4;
  constexpr uint64_t kBStep = BMN ? (2048u >> 4) : (32u >> 4);
  if (nks == 4) {
    mma_f16_ss_x4(lead, d, adesc, bdesc, kAStep, kBStep, idesc, first ? 0u : 1u);
  } else {
    for (int ks = 0; ks < nks; ++ks)
      mma_f16_ss(lead, d, adesc + ks * kAStep, bdesc + ks * kBStep, idesc,
                 (first && ks == 0) ? 0u : 1u);
  }
}

// GEMM1 chunk with A (= P) in TMEM: 8 packed columns per 16-wide K step.
template <bool BMN>
__device__ __forceinline__ void issue_chunk_ts(uint32_t lead, uint32_t d, uint32_t a_tmem,
                                               uint64_t bdesc, uint32_t idesc, int nks,
                                               bool first) {
  constexpr uint64_t kBStep = BMN ? (2048u >> 4) : (32u >> 4);
  for (int ks = 0; ks < nks; ++ks)
    mma_f16_ts(lead, d, a_tmem + 8u * ks, bdesc + ks * kBStep, idesc,
               (first && ks == 0) ? 0u : 1u);
}

template <int MODE, bool A4D, bool W0MN, bool W1MN, bool BF16, bool WIDE, bool PAIR, bool NOPAIR,
          bool W0RES, bool TWO>
__device__ void mma_role(const ChainParams& p, uint32_t base, uint32_t bars, uint32_t tmem_base,
                         volatile uint32_t* abort_flag, int issuer = 0) {
  const bool resident = !PAIR && p.resident != 0;   // (as in the producer)
  // two issuers: issuer 0 takes even tiles, 1 odd ones, each in its own sub-ring
  const bool two = two_issuers(MODE, TWO) && p.two_issuers != 0;
  const uint32_t idesc0 = idesc_f16_f32(BF16 ? 1u : 0u, W0MN ? 1u : 0u, kBlockM, p.N0p);
  const uint32_t idesc1 = idesc_f16_f32(BF16 ? 1u : 0u, W1MN ? 1u : 0u, kBlockM, p.N1p);
  bool ok = true;
  const uint32_t lead = elect_one();
  // slots 0..2: the kernel's entry, setup and dependency events (the second issuer does
  // not record)
  Tracer trace(p, 1, issuer == 0 ? lead : 0u, 3);
  if (resident)
    ok = warp_mbar_wait(bars + 8u * BAR_WFULL, 0u, p, abort_flag, SITE_MMA_WEIGHTS, 0);
  bool bias_ready = false;   // the epilogue warps write the bias operands at the start

  // Descriptors of every operand region, built once; a ring stage / weight chunk / P
  // chunk is then a multiple of its byte size (in 16-byte units) added to them.
  const uint32_t w0_lbo = W0MN ? 8192u : 16u, w1_lbo = W1MN ? 8192u : 16u;
  const uint64_t ring_a = sdesc_sw128(base + p.off_ring, 16u, 1024u);
  const uint64_t ring_w0 = sdesc_sw128(base + p.off_ring + kABytes, w0_lbo, 1024u);
  const uint64_t ring_w1 = sdesc_sw128(base + p.off_ring, w1_lbo, 1024u);
  const uint64_t res_w0 = sdesc_sw128(base + p.off_w0, w0_lbo, 1024u);
  const uint64_t res_w1 = sdesc_sw128(base + p.off_w1, w1_lbo, 1024u);
  const uint64_t p_desc0 = sdesc_sw128(base + p.off_p[0], 16u, 1024u);
  // Bias step operands (see fill_bias_operands): B is MN-major whatever the weights are.
  const uint32_t ones_addr = base + p.off_bias;
  const uint32_t n0blk = static_cast<uint32_t>((p.N0p + 63) >> 6);
  const uint64_t ones_desc = sdesc_sw128(ones_addr, 16u, 0u);
  const uint64_t bias0_desc = sdesc_sw128(ones_addr + kOnesBytes, kBiasBlockBytes, 1024u);
  const uint64_t bias1_desc =
      sdesc_sw128(ones_addr + kOnesBytes + n0blk * kBiasBlockBytes, kBiasBlockBytes, 1024u);
  const uint32_t idesc_b0 = idesc_f16_f32(BF16 ? 1u : 0u, 1u, kBlockM, p.N0p);
  const uint32_t idesc_b1 = idesc_f16_f32(BF16 ? 1u : 0u, 1u, kBlockM, p.N1p);
  const uint32_t stage_step = p.stage_bytes >> 4;
  const uint32_t w0_step = p.w0_chunk_bytes >> 4, w1_step = p.w1_chunk_bytes >> 4;
  // K steps of GEMM0's chunks: full (4) except the last channel block of each tap / the
  // last chunk of K0.
  const int last_rem = p.K0 - (p.kc_per_tap - 1) * kChunkK;
  const int last_nks = last_rem >= 64 ? 4 : (last_rem + 15) >> 4;
  const int rem1 = p.N0p - (p.kchunks1 - 1) * kChunkK;
  const int last_nks1 = rem1 >= 64 ? 4 : (rem1 >> 4);
  // Wide chains: GEMM0 in two passes of N = 256 and N0p - 256 (the halves of N0), each
  // with its bias four 64-wide blocks apart.  (A separate instantiation, WIDE, so that no
  // other launch pays for them.)
  const uint32_t idesc0_lo = WIDE ? idesc_f16_f32(BF16 ? 1u : 0u, W0MN ? 1u : 0u, kBlockM, 256) : 0u;
  const uint32_t idesc0_hi =
      WIDE ? idesc_f16_f32(BF16 ? 1u : 0u, W0MN ? 1u : 0u, kBlockM, p.N0p - 256) : 0u;
  const uint32_t idesc_b0_lo = WIDE ? idesc_f16_f32(BF16 ? 1u : 0u, 1u, kBlockM, 256) : 0u;
  const uint32_t idesc_b0_hi = WIDE ? idesc_f16_f32(BF16 ? 1u : 0u, 1u, kBlockM, p.N0p - 256) : 0u;
  // Three-operator chain: GEMM2 reads P1 (K-major, as P) and the resident W2 (MN-major).
  // Other modes never read these (zero, so that they cost nothing).
  constexpr bool kThree = MODE == MODE_CHAIN3;
  const uint32_t idesc2 = kThree ? idesc_f16_f32(BF16 ? 1u : 0u, 1u, kBlockM, p.N2p) : 0u;
  const uint64_t p1_desc0 = kThree ? sdesc_sw128(base + p.off_p1[0], 16u, 1024u) : 0u;
  const uint64_t res_w2 = kThree ? sdesc_sw128(base + p.off_w2, 8192u, 1024u) : 0u;
  const uint32_t n1blk = static_cast<uint32_t>((p.N1p + 63) >> 6);
  const uint64_t bias2_desc =
      kThree ? sdesc_sw128(ones_addr + kOnesBytes + (n0blk + n1blk) * kBiasBlockBytes,
                           kBiasBlockBytes, 1024u)
             : 0u;
  const uint32_t idesc_b2 = kThree ? idesc_f16_f32(BF16 ? 1u : 0u, 1u, kBlockM, p.N2p) : 0u;
  const uint32_t w2_step = kThree ? p.w2_chunk_bytes >> 4 : 0u;
  const int rem2 = kThree ? p.N1p - (p.kchunks2 - 1) * kChunkK : 64;
  const int last_nks2 = rem2 >= 64 ? 4 : (rem2 >> 4);

  int stage = 0;
  uint32_t phase = 0;
  SubRing sr = subring_of(p, issuer);   // two issuers: this issuer's sub-ring
  const int ntiles = local_tiles(p);
  trace(EV_MMA_SETUP, 0, 0);
  // The setup above overlaps the previous grid's tail; no bounded wait below runs while
  // that grid is pending.
  grid_dependency_wait();
  trace(EV_DEP_READY, 0, 0);

  // GEMM0 of the it-th tile: D0[b] = A . W0 over all K chunks; commits ACC_FULL[b].
  auto issue_g0 = [&](int it) -> bool {
    const int32_t t = blockIdx.x + it * gridDim.x;
    const uint32_t b = buf_of(p, it);

    if ((MODE != MODE_CHAIN && MODE != MODE_CHAIN3) || PAIR || (!NOPAIR && p.p_tmem && !two)) {
      // The epilogue must have drained the buffer's previous tile (with P in TMEM: its
      // GEMM1 accumulator, the last thing read from the buffer).  (A chain with two
      // issuers keeps P and D1 apart from D0: D0 was drained before that tile's P was
      // published, which its GEMM1, issued before this GEMM0, waited for.)
      if (!warp_mbar_wait(bars + 8u * (BAR_ACC_EMPTY0 + b), use_of(p, it) ^ 1u, p, abort_flag,
                          SITE_MMA_ACC_EMPTY, t))
        return false;
      trace(EV_MMA_ACC_FREE, b, it);
      // Orders these MMAs after the epilogue's TMEM reads of the buffer.  This fence costs
      // hundreds of cycles while earlier MMAs are in flight, so it is taken once per tile,
      // only where the wait synchronised with tcgen05 operations of another thread.
      tc_fence_after_sync();
    }
    const uint32_t d0 = tmem_base + p.d0_col[b];
    int cb = 0;       // channel block within the tap (4-D) / chunk index (2-D)
    int s_tap = 0;    // halo: the column tap of the stage
    for (int kc = 0; kc < p.kstages0; ++kc) {
      if (two) {   // this issuer's sub-ring
        stage = sr.slot;
        phase = sr.phase;
        advance_subring(sr);
      }
      trace(EV_MMA_WAIT, kc, it);
      if (!warp_mbar_wait(bars + 8u * (BAR_FULL0 + stage), phase, p, abort_flag, SITE_MMA_FULL, t))
        return false;
      trace(EV_MMA_FULL, kc, it);   // TMA data: no tcgen05 ordering needed
      const uint64_t adesc = ring_a + static_cast<uint64_t>(stage) * stage_step;
      const int nks = cb == p.kc_per_tap - 1 ? last_nks : 4;
      if (A4D && p.halo) {
        // The stage holds rows ho0 - pad .. + 8 + R - 1 (16 pixels each): row tap r starts
        // 16 rows = 2 KiB (two swizzle atoms) further in.
        for (int r = 0; r < p.R; ++r) {
          const int wchunk = (r * p.S + s_tap) * p.kc_per_tap + cb;
          issue_chunk<W0MN>(lead, d0, adesc + static_cast<uint64_t>(r) * (2048u >> 4),
                            res_w0 + static_cast<uint64_t>(wchunk) * w0_step, idesc0, nks,
                            kc == 0 && r == 0);
        }
        if (++cb == p.kc_per_tap) { cb = 0; ++s_tap; }
      } else {
        if (W0RES && it == 0) {
          // the resident W0's chunk kc has landed (once per CTA; TMA data, no tcgen05 order)
          if (!warp_mbar_wait(bars + 8u * (BAR_W0C0 + kc), 0u, p, abort_flag, SITE_MMA_WEIGHTS, t))
            return false;
        }
        const uint64_t bdesc = (resident || W0RES)
                                   ? res_w0 + static_cast<uint64_t>(kc) * w0_step
                                   : ring_w0 + static_cast<uint64_t>(stage) * stage_step;
        if (++cb == p.kc_per_tap) cb = 0;
        issue_chunk<W0MN>(lead, d0, adesc, bdesc, idesc0, nks, kc == 0);
      }
      trace(EV_MMA_ISSUED, kc, it);
      mma_commit(lead, bars + 8u * (BAR_EMPTY0 + stage));   // frees the ring slot when read
      if (++stage == static_cast<int>(p.num_stages)) { stage = 0; phase ^= 1u; }
    }
    // The bias step comes last, so the epilogue warps' first write of its operands
    // overlaps the first tile's MMAs.
    if (!bias_ready) {
      if (!warp_mbar_wait(bars + 8u * BAR_BIAS_READY, 0u, p, abort_flag, SITE_MMA_WEIGHTS, t))
        return false;
      bias_ready = true;
    }
    mma_f16_ss(lead, d0, ones_desc, bias0_desc, idesc_b0, 1u);   // D0 += bias
    mma_commit(lead, bars + 8u * (BAR_ACC_FULL0 + b));
    trace(EV_MMA_G0_DONE, b, it);
    return true;
  };

  // GEMM1 of the j-th tile: D1[b] = P[b] . W1, P[b] being the epilogue's fp16/bf16 tile.
  auto issue_g1 = [&](int j) -> bool {
    const int32_t t = blockIdx.x + j * gridDim.x;
    const uint32_t b = buf_of(p, j);
    if (!warp_mbar_wait(bars + 8u * (BAR_P_FULL0 + b), use_of(p, j), p, abort_flag, SITE_MMA_P_FULL, t))
      return false;
    trace(EV_MMA_P_READY, b, j);
    tc_fence_after_sync();
    const uint32_t d1 = tmem_base + p.d1_col[b];
    const int per = static_cast<int>(p.w1_per_stage);   // streamed W1 chunks per ring stage
    int slot = 0;
    for (int kc1 = 0; kc1 < p.kchunks1; ++kc1) {
      uint64_t bdesc;
      if (resident) {
        bdesc = res_w1 + static_cast<uint64_t>(kc1) * w1_step;
      } else {
        if (slot == 0) {
          if (!warp_mbar_wait(bars + 8u * (BAR_FULL0 + stage), phase, p, abort_flag,
                              SITE_MMA_FULL, t))
            return false;
          trace(EV_MMA_W1_FULL, kc1, j);
        }
        bdesc = ring_w1 + static_cast<uint64_t>(stage) * stage_step +
                static_cast<uint64_t>(slot) * w1_step;
      }
      const int nks1 = kc1 == p.kchunks1 - 1 ? last_nks1 : 4;
      if (PAIR || (!NOPAIR && p.p_tmem)) {
        issue_chunk_ts<W1MN>(lead, d1, tmem_base + p.pt_col[b] + 32u * static_cast<uint32_t>(kc1),
                             bdesc, idesc1, nks1, kc1 == 0);
      } else {
        // P buffer b, chunk kc1 (P buffers are whole 1 KiB multiples apart)
        const uint64_t adesc = p_desc0 + ((p.off_p[b] - p.off_p[0]) >> 4) +
                               static_cast<uint64_t>(kc1) * (kPChunkBytes >> 4);
        issue_chunk<W1MN>(lead, d1, adesc, bdesc, idesc1, nks1, kc1 == 0);
      }
      if (!resident && (++slot == per || kc1 == p.kchunks1 - 1)) {
        slot = 0;
        mma_commit(lead, bars + 8u * (BAR_EMPTY0 + stage));
        if (++stage == static_cast<int>(p.num_stages)) { stage = 0; phase ^= 1u; }
      }
    }
    mma_f16_ss(lead, d1, ones_desc, bias1_desc, idesc_b1, 1u);   // D1 += bias
    mma_commit(lead, bars + 8u * (BAR_D1_FULL0 + b));
    trace(EV_MMA_G1_DONE, b, j);
    return true;
  };

  // GEMM2 of the j-th tile (three-operator chain): D2[b] = P1[b] . W2, both resident in
  // shared memory; commits D2_FULL[b].
  auto issue_g2 = [&](int j) -> bool {
    const int32_t t = blockIdx.x + j * gridDim.x;
    const uint32_t b = buf_of(p, j);
    if (!warp_mbar_wait(bars + 8u * (BAR_P1_FULL0 + b), use_of(p, j), p, abort_flag,
                        SITE_MMA_P1_FULL, t))
      return false;
    tc_fence_after_sync();
    const uint32_t d2 = tmem_base + p.d2_col[b];
    for (int kc2 = 0; kc2 < p.kchunks2; ++kc2) {
      const uint64_t adesc = p1_desc0 + ((p.off_p1[b] - p.off_p1[0]) >> 4) +
                             static_cast<uint64_t>(kc2) * (kPChunkBytes >> 4);
      const uint64_t bdesc = res_w2 + static_cast<uint64_t>(kc2) * w2_step;
      issue_chunk<true>(lead, d2, adesc, bdesc, idesc2, kc2 == p.kchunks2 - 1 ? last_nks2 : 4,
                        kc2 == 0);
    }
    mma_f16_ss(lead, d2, ones_desc, bias2_desc, idesc_b2, 1u);   // D2 += bias
    mma_commit(lead, bars + 8u * (BAR_D2_FULL0 + b));
    trace(EV_MMA_G2_DONE, b, j);
    return true;
  };

  // GEMM1 of the tiles j and (if `two`) j + 1 from one group of W1 stages (w1_group):
  // the first tile waits for the stages, the second reads the same ones, and the stages
  // are released after both.
  auto issue_g1_pair = [&](int j, bool two) -> bool {
    const int per = static_cast<int>(p.w1_per_stage);
    const int s_first = stage;
    const uint32_t ph_first = phase;
    for (int r = 0; r < (two ? 2 : 1); ++r) {
      const int jj = j + r;
      const int32_t t = blockIdx.x + jj * gridDim.x;
      const uint32_t b = static_cast<uint32_t>(jj & 1), u = static_cast<uint32_t>(jj >> 1);
      if (!warp_mbar_wait(bars + 8u * (BAR_P_FULL0 + b), u & 1u, p, abort_flag, SITE_MMA_P_FULL,
                          t))
        return false;
      trace(EV_MMA_P_READY, b, jj);
      tc_fence_after_sync();
      const uint32_t d1 = tmem_base + p.d1_col[b];
      int s = s_first, slot = 0;
      uint32_t ph = ph_first;
      for (int kc1 = 0; kc1 < p.kchunks1; ++kc1, ++slot) {
        if (slot == per) {
          slot = 0;
          if (++s == static_cast<int>(p.num_stages)) { s = 0; ph ^= 1u; }
        }
        if (r == 0 && slot == 0) {
          if (!warp_mbar_wait(bars + 8u * (BAR_FULL0 + s), ph, p, abort_flag, SITE_MMA_FULL, t))
            return false;
          trace(EV_MMA_W1_FULL, kc1, jj);
        }
        const uint64_t bdesc = ring_w1 + static_cast<uint64_t>(s) * stage_step +
                               static_cast<uint64_t>(slot) * w1_step;
        const int nks1 = kc1 == p.kchunks1 - 1 ? last_nks1 : 4;
        issue_chunk_ts<W1MN>(lead, d1, tmem_base + p.pt_col[b] + 32u * kc1, bdesc, idesc1, nks1,
                             kc1 == 0);
        trace(EV_MMA_ISSUED, 8 + kc1, jj);   // GEMM1 chunks: group 8 + chunk
      }
      mma_f16_ss(lead, d1, ones_desc, bias1_desc, idesc_b1, 1u);   // D1 += bias
      mma_commit(lead, bars + 8u * (BAR_D1_FULL0 + b));
      trace(EV_MMA_G1_DONE, b, jj);
    }
    for (int i = 0; i < (p.kchunks1 + per - 1) / per; ++i) {
      mma_commit(lead, bars + 8u * (BAR_EMPTY0 + stage));
      if (++stage == static_cast<int>(p.num_stages)) { stage = 0; phase ^= 1u; }
    }
    return true;
  };

  // Wide chains, GEMM0 of tile it over half h of N0 into TMEM columns [256h, 256h + 256);
  // commits ACC_FULL[h].  The tile's second pass overwrites the previous tile's D1 (which
  // sits in the other half), so it waits for that tile's epilogue to have drained it.
  auto issue_g0_half = [&](int it, int h, bool second) -> bool {
    const int32_t t = blockIdx.x + it * gridDim.x;
    if (second && it > 0) {
      if (!warp_mbar_wait(bars + 8u * BAR_ACC_EMPTY0, static_cast<uint32_t>(it - 1) & 1u, p,
                          abort_flag, SITE_MMA_ACC_EMPTY, t))
        return false;
      trace(EV_MMA_ACC_FREE, h, it);
      tc_fence_after_sync();
    }
    const uint32_t d0 = tmem_base + 256u * static_cast<uint32_t>(h);
    const uint32_t idesc = h ? idesc0_hi : idesc0_lo;
    for (int kc = 0; kc < p.kchunks0; ++kc) {
      trace(EV_MMA_WAIT, kc, it);
      if (!warp_mbar_wait(bars + 8u * (BAR_FULL0 + stage), phase, p, abort_flag, SITE_MMA_FULL, t))
        return false;
      trace(EV_MMA_FULL, kc, it);
      const uint64_t adesc = ring_a + static_cast<uint64_t>(stage) * stage_step;
      const uint64_t bdesc = ring_w0 + static_cast<uint64_t>(stage) * stage_step;
      issue_chunk<W0MN>(lead, d0, adesc, bdesc, idesc, kc == p.kchunks0 - 1 ? last_nks : 4,
                        kc == 0);
      trace(EV_MMA_ISSUED, kc, it);
      mma_commit(lead, bars + 8u * (BAR_EMPTY0 + stage));
      if (++stage == static_cast<int>(p.num_stages)) { stage = 0; phase ^= 1u; }
    }
    if (!bias_ready) {
      if (!warp_mbar_wait(bars + 8u * BAR_BIAS_READY, 0u, p, abort_flag, SITE_MMA_WEIGHTS, t))
        return false;
      bias_ready = true;
    }
    mma_f16_ss(lead, d0, ones_desc,
               bias0_desc + static_cast<uint64_t>(h) * ((4u * kBiasBlockBytes) >> 4),
               h ? idesc_b0_hi : idesc_b0_lo, 1u);
    mma_commit(lead, bars + 8u * (BAR_ACC_FULL0 + h));
    trace(EV_MMA_G0_DONE, h, it);
    return true;
  };

  // Wide chains, GEMM1 of tile it: D1 (at d1_col[it & 1], the first half's upper columns)
  // = P_f . W1[f] + P_s . W1[s] over the first half f = it & 1, then the other one s, each
  // as soon as its P (packed in place at 256h) is published; commits D1_FULL[0].
  auto issue_g1_wide = [&](int it) -> bool {
    const int32_t t = blockIdx.x + it * gridDim.x;
    const int f = it & 1;
    const uint32_t d1 = tmem_base + p.d1_col[f];
    const int per = static_cast<int>(p.w1_per_stage);
    bool first = true;
    for (int pass = 0; pass < 2; ++pass) {
      const int h = pass == 0 ? f : f ^ 1;
      if (!warp_mbar_wait(bars + 8u * (BAR_P_FULL0 + h), static_cast<uint32_t>(it) & 1u, p,
                          abort_flag, SITE_MMA_P_FULL, t))
        return false;
      trace(EV_MMA_P_READY, h, it);
      tc_fence_after_sync();
      const int kbeg = 4 * h, kend = h == 0 ? min(4, p.kchunks1) : p.kchunks1;
      int slot = 0;
      for (int kc1 = kbeg; kc1 < kend; ++kc1) {
        if (slot == 0) {
          if (!warp_mbar_wait(bars + 8u * (BAR_FULL0 + stage), phase, p, abort_flag,
                              SITE_MMA_FULL, t))
            return false;
          trace(EV_MMA_W1_FULL, kc1, it);
        }
        const uint64_t bdesc = ring_w1 + static_cast<uint64_t>(stage) * stage_step +
                               static_cast<uint64_t>(slot) * w1_step;
        issue_chunk_ts<W1MN>(lead, d1,
                             tmem_base + 256u * static_cast<uint32_t>(h) +
                                 32u * static_cast<uint32_t>(kc1 - kbeg),
                             bdesc, idesc1, kc1 == p.kchunks1 - 1 ? last_nks1 : 4, first);
        first = false;
        if (++slot == per || kc1 == kend - 1) {
          slot = 0;
          mma_commit(lead, bars + 8u * (BAR_EMPTY0 + stage));
          if (++stage == static_cast<int>(p.num_stages)) { stage = 0; phase ^= 1u; }
        }
      }
    }
    mma_f16_ss(lead, d1, ones_desc, bias1_desc, idesc_b1, 1u);   // D1 += bias
    mma_commit(lead, bars + 8u * BAR_D1_FULL0);
    trace(EV_MMA_G1_DONE, 0, it);
    return true;
  };

  if (ok) {
    if constexpr (MODE == MODE_CHAIN && WIDE) {
      // Per tile: GEMM0 over the first half, over the second, then GEMM1.  The next tile's
      // first half is the other one, so its GEMM0 runs while this tile's D1 drains.
      for (int it = 0; ok && it < ntiles; ++it) {
        const int f = it & 1;
        ok = issue_g0_half(it, f, false);
        if (ok) ok = issue_g0_half(it, f ^ 1, true);
        if (ok) ok = issue_g1_wide(it);
      }
    } else if (MODE == MODE_CHAIN && TWO && two) {
      // Two issuers: this one takes the tiles issuer, issuer + 2, ..., each GEMM0 then
      // GEMM1 into buffer `issuer`; while it waits for the epilogue's P, the other issuer's
      // GEMM0 keeps the tensor core busy.
      for (int j = issuer; ok && j < ntiles; j += 2) {
        ok = issue_g0(j);
        if (ok) ok = issue_g1(j);
      }
    } else if (MODE == MODE_CHAIN && (PAIR || (!NOPAIR && p.p_tmem))) {
      // Pairs of tiles: while the epilogue of one tile drains, the other tile's MMAs run.
      for (int it = 0; ok && it < 2 && it < ntiles; ++it) ok = issue_g0(it);
      for (int k = 0; ok && k < ntiles; k += 2) {
        if (p.w1_group) {
          ok = issue_g1_pair(k, k + 1 < ntiles);
        } else {
          ok = issue_g1(k);
          if (ok && k + 1 < ntiles) ok = issue_g1(k + 1);
        }
        if (ok && k + 2 < ntiles) ok = issue_g0(k + 2);
        if (ok && k + 3 < ntiles) ok = issue_g0(k + 3);
      }
    } else if (MODE == MODE_CHAIN3) {
      // Pairs of tiles, each GEMM for both tiles before the next GEMM: while one tile's
      // epilogue drains an accumulator, the other tile's MMAs run.  Buffer b's D0, D1, D2
      // and P0, P1 are free again for tile k + 2 because the group that drains them works
      // through its tiles in order and the MMAs complete in issue order.
      for (int k = 0; ok && k < ntiles; k += 2) {
        const bool two = k + 1 < ntiles;
        ok = issue_g0(k);
        if (ok && two) ok = issue_g0(k + 1);
        if (ok) ok = issue_g1(k);
        if (ok && two) ok = issue_g1(k + 1);
        if (ok) ok = issue_g2(k);
        if (ok && two) ok = issue_g2(k + 1);
      }
    } else if (MODE == MODE_CHAIN) {
      // A D0 buffer is free again once the epilogue has published that tile's P, so
      // G0(j+L) follows G1(j); with L buffers, L tiles are in flight.
      const int L = 1 << p.nbuf_log2;
      for (int it = 0; ok && it < L && it < ntiles; ++it) ok = issue_g0(it);
      for (int j = 0; ok && j < ntiles; ++j) {
        ok = issue_g1(j);
        if (ok && j + L < ntiles) ok = issue_g0(j + L);
      }
    } else {
      for (int it = two ? issuer : 0; ok && it < ntiles; it += two ? 2 : 1) ok = issue_g0(it);
    }
  }
  // Whatever happened, no MMA may still be running when TMEM is released (with two
  // issuers the barrier counts both commits).
  mma_commit(lead, bars + 8u * BAR_MMA_DONE);
  (void)mbar_wait(bars + 8u * BAR_MMA_DONE, 0u, p.wait_limit_ns, nullptr, p.err, p.kernel_id,
                  SITE_MMA_DRAIN, 0);
  __syncwarp();
}

// ------------------------------------------------------------------------------------
// epilogue (4 warps, one TMEM lane = one tile row per thread)
// ------------------------------------------------------------------------------------
template <int ACT>
__device__ __forceinline__ float act_fn(float x) {
  // hardswish(x) = x * min(max(x + 3, 0), 6) / 6 = x * clamp(x / 6 + 1/2, 0, 1):
  // one fused multiply-add with saturation and one multiply.
  if constexpr (ACT == 2) return x * __saturatef(fmaf(x, 1.0f / 6.0f, 0.5f));
  return x;
}

// Two fp32 values -> one packed fp16/bf16 pair (lo in the low half), round to nearest
// even; RELU clamps negative results to zero in the same conversion.
template <bool BF16, bool RELU>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  if constexpr (BF16 && RELU)
    asm("cvt.rn.relu.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  else if constexpr (BF16)
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  else if constexpr (RELU)
    asm("cvt.rn.relu.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Stores 16 consecutive columns [c0, c0+16) of row `row` into a K-major, 128B-swizzled
// tile: 64-column chunks of `chunk_bytes`, 128 B per row, and the 16-byte unit j of row r
// stored at unit j ^ (r & 7) -- the layout TMA writes with SWIZZLE_128B and tcgen05
// reads through a SWIZZLE_128B descriptor.
__device__ __forceinline__ void st_row16_sw128(uint32_t tile, int row, int c0,
                                               uint32_t chunk_bytes, const uint32_t (&v)[8]) {
  const uint32_t chunk = static_cast<uint32_t>(c0) >> 6;
  const uint32_t j = (static_cast<uint32_t>(c0) & 63u) >> 3;
  const uint32_t rb = tile + chunk * chunk_bytes + static_cast<uint32_t>(row) * 128u;
  const uint32_t x = static_cast<uint32_t>(row) & 7u;
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(rb + ((j ^ x) << 4)), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3])
               : "memory");
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(rb + (((j + 1) ^ x) << 4)),
               "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// 16 accumulator columns (the bias is already in them) -> act -> 8 packed pairs.
template <bool BF16, int ACT>
__device__ __forceinline__ void convert16(const uint32_t (&r)[16], uint32_t (&out)[8]) {
#pragma unroll
  for (int j = 0; j < 8; ++j)
    out[j] = pack2<BF16, ACT == 1>(act_fn<ACT>(__uint_as_float(r[2 * j])),
                                   act_fn<ACT>(__uint_as_float(r[2 * j + 1])));
}

// The drains below walk a row's TMEM columns in steps of 32: both 16-column loads of a
// step are issued together and waited for once, then converted.  This plain loop (no
// loads carried across iterations, no early exits) measured faster than a software-
// pipelined one whose exits depend on the run-time column count.  The drains are called,
// not inlined: one inlined copy per activation pushed the kernel past its register
// budget (168 per thread with ten warps) and made it spill.

// TMEM columns of this thread's row -> act -> dtype -> K-major 128B-swizzled smem
// tile.  The 32-column blocks c_first, c_first + c_step, ... below ncols (c_step = 32:
// all columns; 64: every other block).  ncols is a multiple of 16.
template <bool BF16, int ACT>
__device__ __noinline__ void drain_to_smem_act(uint32_t tm_lane, uint32_t col0, int c_first,
                                                  int c_step, int ncols, uint32_t tile,
                                                  int row, uint32_t chunk_bytes) {
  for (int c = c_first; c < ncols; c += c_step) {
    const bool two = c + 16 < ncols;
    uint32_t a[16], b[16], v[8];
    tmem_ld32(tm_lane + col0 + c, two, a, b);
    tmem_wait_ld(a, b);
    convert16<BF16, ACT>(a, v);
    st_row16_sw128(tile, row, c, chunk_bytes, v);
    if (two) {
      convert16<BF16, ACT>(b, v);
      st_row16_sw128(tile, row, c + 16, chunk_bytes, v);
    }
  }
}

template <bool BF16>
__device__ __forceinline__ void drain_to_smem(int act, uint32_t tm_lane, uint32_t col0,
                                              int c_first, int c_step, int ncols, uint32_t tile,
                                              int row, uint32_t chunk_bytes) {
  if (act == 2)
    drain_to_smem_act<BF16, 2>(tm_lane, col0, c_first, c_step, ncols, tile, row, chunk_bytes);
  else if (act == 1)
    drain_to_smem_act<BF16, 1>(tm_lane, col0, c_first, c_step, ncols, tile, row, chunk_bytes);
  else
    drain_to_smem_act<BF16, 0>(tm_lane, col0, c_first, c_step, ncols, tile, row, chunk_bytes);
}

// GEMM0 accumulator columns [col0, col0 + ncols) of this thread's row -> act -> dtype -> packed pairs written back into TMEM at p_col0 + c / 2.  With p_col0 = col0, P
// overwrites columns of D0 this thread has already read: the step at c writes columns
// below col0 + c / 2 + 16 <= col0 + c + 32, the next step's first column.  Valid only
// when one warpgroup owns the whole row.
template <bool BF16, int ACT>
__device__ __noinline__ void drain_to_tmem_act(uint32_t tm_lane, uint32_t col0, int ncols,
                                                  uint32_t p_col0) {
  for (int c = 0; c < ncols; c += 32) {
    const bool two = c + 16 < ncols;
    uint32_t a[16], b[16], v[8];
    tmem_ld32(tm_lane + col0 + c, two, a, b);
    tmem_wait_ld(a, b);
    convert16<BF16, ACT>(a, v);
    tmem_st8(tm_lane + p_col0 + (c >> 1), v);
    if (two) {
      convert16<BF16, ACT>(b, v);
      tmem_st8(tm_lane + p_col0 + ((c + 16) >> 1), v);
    }
  }
  tmem_wait_st();
}

template <bool BF16>
__device__ __forceinline__ void drain_to_tmem(int act, uint32_t tm_lane, uint32_t col0,
                                              int ncols, uint32_t p_col0) {
  if (act == 2)
    drain_to_tmem_act<BF16, 2>(tm_lane, col0, ncols, p_col0);
  else if (act == 1)
    drain_to_tmem_act<BF16, 1>(tm_lane, col0, ncols, p_col0);
  else
    drain_to_tmem_act<BF16, 0>(tm_lane, col0, ncols, p_col0);
}

// 16 converted columns (8 packed pairs) to global memory at `dst`, 16 bytes at a time;
// `n` = the columns left in the row (units at or past the row's end are not stored).
__device__ __forceinline__ void st_global_cols16(uint8_t* dst, const uint32_t (&v)[8], int n) {
  if (n >= 8)
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "r"(v[0]), "r"(v[1]),
                 "r"(v[2]), "r"(v[3])
                 : "memory");
  if (n >= 16)
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 16), "r"(v[4]),
                 "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

// Accumulator columns [col0, col0 + ncols) of this thread's row -> act -> dtype -> the
// row in global memory (`dst` = its first element), with no staging tile.  Columns at or
// past `nvalid` (the output's width, a multiple of 8) and a row outside the output
// (`row_ok` false: the last tile's rows past M) are not stored.  The TMEM loads are
// warp-collective, so every lane runs the loop.
template <bool BF16, int ACT>
__device__ __noinline__ void drain_to_global_act(uint32_t tm_lane, uint32_t col0, int ncols,
                                                    uint8_t* dst, int nvalid, bool row_ok) {
  for (int c = 0; c < ncols; c += 32) {
    const bool two = c + 16 < ncols;
    uint32_t a[16], b[16], v[8];
    tmem_ld32(tm_lane + col0 + c, two, a, b);
    tmem_wait_ld(a, b);
    if (row_ok) {
      convert16<BF16, ACT>(a, v);
      st_global_cols16(dst + 2 * c, v, nvalid - c);
      if (two) {
        convert16<BF16, ACT>(b, v);
        st_global_cols16(dst + 2 * (c + 16), v, nvalid - c - 16);
      }
    }
  }
}

template <bool BF16>
__device__ __forceinline__ void drain_to_global(int act, uint32_t tm_lane, uint32_t col0,
                                                int ncols, uint8_t* dst, int nvalid, bool row_ok) {
  if (act == 2)
    drain_to_global_act<BF16, 2>(tm_lane, col0, ncols, dst, nvalid, row_ok);
  else if (act == 1)
    drain_to_global_act<BF16, 1>(tm_lane, col0, ncols, dst, nvalid, row_ok);
  else
    drain_to_global_act<BF16, 0>(tm_lane, col0, ncols, dst, nvalid, row_ok);
}

// Accumulator columns [col0, col0 + ncols) of this thread's row (one output pixel) ->
// act -> dtype -> the output, 16 columns at a time through the warp's 1 KiB slot (32 rows
// x 32 B, row = lane): one TMA store per step of 16 channels x 16 x 2 pixels at (c, wo0, h0,
// n), the warp's two output rows; lane 0 first waits until its previous store has read the
// slot.  Columns at or past `nvalid` are not stored, nor anything if `store` is false (both
// rows below the image; TMA clips the rest).  A small slot and short steps keep the kernel
// within its 168-register cap, and TMA writes whole 32-byte sectors where stores from
// registers (one lane per pixel, 256 bytes apart) take a cache line per lane.
template <bool BF16, int ACT>
__device__ __noinline__ void drain16_to_slot_act(uint32_t tm_lane, uint32_t col0, int ncols,
                                                 int nvalid, uint32_t slot, const CUtensorMap* map,
                                                 int32_t wo0, int32_t h0, int32_t n, bool store,
                                                 int lane) {
  const uint32_t rb = slot + static_cast<uint32_t>(lane) * 32u;
  for (int c = 0; c < ncols; c += 16) {
    uint32_t a[16], v[8];
    tmem_ld16(tm_lane + col0 + c, a);
    tmem_wait_ld(a);
    convert16<BF16, ACT>(a, v);
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(rb), "r"(v[0]), "r"(v[1]),
                 "r"(v[2]), "r"(v[3])
                 : "memory");
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(rb + 16u), "r"(v[4]),
                 "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && store && c < nvalid) {
      tma_store_4d(map, slot, c, wo0, h0, n);
      bulk_commit_group();
    }
  }
}

template <bool BF16>
__device__ __forceinline__ void drain16_to_slot(int act, uint32_t tm_lane, uint32_t col0,
                                                int ncols, int nvalid, uint32_t slot,
                                                const CUtensorMap* map, int32_t wo0, int32_t h0,
                                                int32_t n, bool store, int lane) {
  if (act == 2)
    drain16_to_slot_act<BF16, 2>(tm_lane, col0, ncols, nvalid, slot, map, wo0, h0, n, store, lane);
  else if (act == 1)
    drain16_to_slot_act<BF16, 1>(tm_lane, col0, ncols, nvalid, slot, map, wo0, h0, n, store, lane);
  else
    drain16_to_slot_act<BF16, 0>(tm_lane, col0, ncols, nvalid, slot, map, wo0, h0, n, store, lane);
}

// ------------------------------------------------------------------------------------
// wide drains: 64 accumulator columns per TMEM load and wait
// ------------------------------------------------------------------------------------
// Waits for this thread's outstanding TMEM loads and ties all 64 loaded registers to the
// wait, so that none of their uses is scheduled before it.
__device__ __forceinline__ void tmem_wait_ld64(uint32_t (&r)[64]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
  asm volatile(""
               : "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]), "+r"(r[36]), "+r"(r[37]),
                 "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]), "+r"(r[42]), "+r"(r[43]),
                 "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]), "+r"(r[48]), "+r"(r[49]),
                 "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), "+r"(r[55]),
                 "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), "+r"(r[61]),
                 "+r"(r[62]), "+r"(r[63])
               :
               : "memory");
}

// As drain_to_tmem_act (GEMM0's accumulator -> act -> packed pairs written back over the
// columns already read), 64 columns per load (ncols a multiple of 64) and 32 packed
// columns per store: step c writes columns below p_col0 + c / 2 + 32 <= col0 + c + 64,
// the next step's first column, when p_col0 = col0.
template <bool BF16, int ACT>
__device__ __noinline__ void drain64_to_tmem_act(uint32_t tm_lane, uint32_t col0, int ncols,
                                                    uint32_t p_col0) {
  for (int c = 0; c < ncols; c += 64) {
    uint32_t r[64], v[32];
    tmem_ld64x(tm_lane + col0 + c, r);
    tmem_wait_ld64(r);
#pragma unroll
    for (int j = 0; j < 32; ++j)
      v[j] = pack2<BF16, ACT == 1>(act_fn<ACT>(__uint_as_float(r[2 * j])),
                                   act_fn<ACT>(__uint_as_float(r[2 * j + 1])));
    tmem_st32(tm_lane + p_col0 + (c >> 1), v);
  }
  tmem_wait_st();
}

template <bool BF16>
__device__ __forceinline__ void drain64_to_tmem(int act, uint32_t tm_lane, uint32_t col0,
                                                int ncols, uint32_t p_col0) {
  if (act == 2)
    drain64_to_tmem_act<BF16, 2>(tm_lane, col0, ncols, p_col0);
  else if (act == 1)
    drain64_to_tmem_act<BF16, 1>(tm_lane, col0, ncols, p_col0);
  else
    drain64_to_tmem_act<BF16, 0>(tm_lane, col0, ncols, p_col0);
}

// 64 accumulator columns of this thread's row (TMEM address taddr) -> act -> dtype -> row
// `row` of a 128 x 64 staging tile in the 128B-swizzled layout a TMA store reads.
template <bool BF16, int ACT>
__device__ __noinline__ void drain64_to_staging_act(uint32_t taddr, uint32_t staging, int row) {
  uint32_t r[64];
  tmem_ld64x(taddr, r);
  tmem_wait_ld64(r);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      v[k] = pack2<BF16, ACT == 1>(act_fn<ACT>(__uint_as_float(r[16 * j + 2 * k])),
                                   act_fn<ACT>(__uint_as_float(r[16 * j + 2 * k + 1])));
    st_row16_sw128(staging, row, 16 * j, kPChunkBytes, v);
  }
}

template <bool BF16>
__device__ __forceinline__ void drain64_to_staging(int act, uint32_t taddr, uint32_t staging,
                                                   int row) {
  if (act == 2)
    drain64_to_staging_act<BF16, 2>(taddr, staging, row);
  else if (act == 1)
    drain64_to_staging_act<BF16, 1>(taddr, staging, row);
  else
    drain64_to_staging_act<BF16, 0>(taddr, staging, row);
}

// Exchanges 16-byte units inside each quad of lanes (lanes 4q .. 4q + 3): on entry lane
// 4q + i holds units 0..3 (x[u][0..3]) of row 4q + i of the warp's rows; on return it holds
// unit i of rows 4q + 0 .. 4q + 3 (x[j] = unit i of row 4q + j), so that the quad's four
// lanes together hold one row's 64 contiguous bytes per j.  Two rounds of lane-xor
// exchanges, one per bit of the lane index within the quad: in the round for bit b, a lane
// swaps with lane ^ (1 << b) every unit u whose bit b differs from its own lane bit.
__device__ __forceinline__ void quad_transpose_units(uint32_t (&x)[4][4], int lane) {
  const bool i0 = (lane & 1) != 0, i1 = (lane & 2) != 0;
#pragma unroll
  for (int m = 0; m < 2; ++m) {          // bit 0: units 2m and 2m + 1
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t send = i0 ? x[2 * m][k] : x[2 * m + 1][k];
      const uint32_t got = __shfl_xor_sync(0xffffffffu, send, 1);
      if (i0) x[2 * m][k] = got; else x[2 * m + 1][k] = got;
    }
  }
#pragma unroll
  for (int m = 0; m < 2; ++m) {          // bit 1: units m and m + 2
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t send = i1 ? x[m][k] : x[m + 2][k];
      const uint32_t got = __shfl_xor_sync(0xffffffffu, send, 2);
      if (i1) x[m][k] = got; else x[m + 2][k] = got;
    }
  }
}

// GEMM1's accumulator columns [col0, col0 + ncols) of the warp's 32 rows -> act -> dtype ->
// global memory, 64 columns per wait (ncols a multiple of 64) and coalesced: after
// quad_transpose_units each store instruction of the warp writes eight rows' 64
// contiguous bytes.  `out_row0` is the warp's first row in the output (`rows` valid rows
// in all, `ld` elements per row), `nvalid` the output's width (a multiple of 8); rows and
// 16-byte units outside the output are not stored.  Every lane runs the loop
// (warp-collective loads and shuffles).
template <bool BF16, int ACT>
__device__ __noinline__ void drain64_to_global_act(uint32_t tm_lane, uint32_t col0, int ncols,
                                                      uint8_t* out, int64_t out_row0,
                                                      int64_t rows, int ld, int nvalid,
                                                      int lane);

// Ties 64 more registers, loaded by tcgen05.ld before a tmem_wait_ld64 that has returned,
// to that wait (so that none of their uses is scheduled before it).
__device__ __forceinline__ void tmem_tie64(uint32_t (&r)[64]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
  asm volatile(""
               : "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]), "+r"(r[36]), "+r"(r[37]),
                 "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]), "+r"(r[42]), "+r"(r[43]),
                 "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]), "+r"(r[48]), "+r"(r[49]),
                 "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), "+r"(r[55]),
                 "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), "+r"(r[61]),
                 "+r"(r[62]), "+r"(r[63])
               :
               : "memory");
}

// 64 loaded accumulator columns (registers r) -> act -> dtype: 32 packed pairs.
template <bool BF16, int ACT>
__device__ __forceinline__ void pack64(const uint32_t (&r)[64], uint32_t (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 32; ++j)
    v[j] = pack2<BF16, ACT == 1>(act_fn<ACT>(__uint_as_float(r[2 * j])),
                                 act_fn<ACT>(__uint_as_float(r[2 * j + 1])));
}

// 64 packed output columns of this lane's row (v; output columns from col_base) -> global
// memory: after quad_transpose_units each store instruction of the warp writes eight rows'
// 64 contiguous bytes.
__device__ __forceinline__ void store_packed64(const uint32_t (&v)[32], int col_base, uint8_t* out,
                                               int64_t out_row0, int64_t rows, int ld,
                                               int nvalid, int lane) {
  const int quad = lane >> 2, unit = lane & 3;
#pragma unroll
  for (int h = 0; h < 2; ++h) {        // 32 columns: units of 8 columns, 4 per row
    uint32_t x[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int k = 0; k < 4; ++k) x[u][k] = v[16 * h + 4 * u + k];
    quad_transpose_units(x, lane);
    const int col = col_base + 32 * h + 8 * unit;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t row = out_row0 + 4 * quad + j;
      if (row < rows && col < nvalid)
        asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(
                         out + (static_cast<size_t>(row) * static_cast<size_t>(ld) +
                                static_cast<size_t>(col)) * 2u),
                     "r"(x[j][0]), "r"(x[j][1]), "r"(x[j][2]), "r"(x[j][3])
                     : "memory");
    }
  }
}

template <bool BF16, int ACT>
__device__ __forceinline__ void store64_to_global(const uint32_t (&r)[64], int col_base,
                                                  uint8_t* out, int64_t out_row0, int64_t rows,
                                                  int ld, int nvalid, int lane) {
  uint32_t v[32];
  pack64<BF16, ACT>(r, v);
  store_packed64(v, col_base, out, out_row0, rows, ld, nvalid, lane);
}

template <bool BF16, int ACT>
__device__ __noinline__ void drain64_to_global_act(uint32_t tm_lane, uint32_t col0, int ncols,
                                                      uint8_t* out, int64_t out_row0,
                                                      int64_t rows, int ld, int nvalid,
                                                      int lane) {
  for (int c = 0; c < ncols; c += 64) {
    uint32_t r[64];
    tmem_ld64x(tm_lane + col0 + c, r);
    tmem_wait_ld64(r);
    store64_to_global<BF16, ACT>(r, c, out, out_row0, rows, ld, nvalid, lane);
  }
}

// As drain64_to_global_act, releasing the accumulator early: the last 128 columns (ncols a
// multiple of 64, at least 128) are loaded from TMEM together, and once that load has
// completed -- before any of them is converted or stored -- the warp's lane 0 arrives on
// `release` (a barrier address in the cluster's shared window; the caller's barrier
// counts one arrive per warp) after `tcgen05.fence::before_thread_sync`.  The MMA issuer
// may then overwrite the columns while this warp finishes its stores from registers.
template <bool BF16, int ACT>
__device__ __noinline__ void drain64_release_to_global_act(uint32_t tm_lane, uint32_t col0,
                                                           int ncols, uint8_t* out,
                                                           int64_t out_row0, int64_t rows, int ld,
                                                           int nvalid, int lane,
                                                           uint32_t release) {
  const int head = ncols - 128;   // columns drained before the last 128
  for (int c = 0; c < head; c += 64) {
    uint32_t r[64];
    tmem_ld64x(tm_lane + col0 + c, r);
    tmem_wait_ld64(r);
    store64_to_global<BF16, ACT>(r, c, out, out_row0, rows, ld, nvalid, lane);
  }
  uint32_t r0[64], r1[64];
  tmem_ld64x(tm_lane + col0 + head, r0);
  tmem_ld64x(tm_lane + col0 + head + 64, r1);
  tmem_wait_ld64(r0);
  tmem_tie64(r1);
  tc_fence_before_sync();
  __syncwarp();
  if (lane == 0) mbar_arrive_remote(release);
  uint32_t v0[32], v1[32];
  pack64<BF16, ACT>(r0, v0);
  pack64<BF16, ACT>(r1, v1);
  store_packed64(v0, head, out, out_row0, rows, ld, nvalid, lane);
  store_packed64(v1, head + 64, out, out_row0, rows, ld, nvalid, lane);
}

// 64 packed output columns of this lane's row (v) -> the warp's staging slot (32 rows x
// 128 B, 128B-swizzled: the output map's box of 64 columns x 32 rows) -> one TMA store at
// output column `col`, rows row0 .. row0 + 31 (TMA clips rows past the output; a box whose
// rows all lie past it is not issued), marked evict-first in L2 (the output is not read
// again here; measured ~1 % faster on the FFN-like chain over CTA pairs).  Lane 0 first
// waits until its previous store has read the slot.
__device__ __forceinline__ void stage_store64(const uint32_t (&v)[32], uint32_t slot,
                                              const CUtensorMap* map, int col, int32_t row0,
                                              int64_t rows, int lane) {
  if (lane == 0) bulk_wait_read_all();
  __syncwarp();
  const uint32_t rb = slot + static_cast<uint32_t>(lane) * 128u;
  const uint32_t x = static_cast<uint32_t>(lane) & 7u;
#pragma unroll
  for (uint32_t j = 0; j < 8; ++j)
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(rb + ((j ^ x) << 4)),
                 "r"(v[4 * j]), "r"(v[4 * j + 1]), "r"(v[4 * j + 2]), "r"(v[4 * j + 3])
                 : "memory");
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0 && row0 < rows) {
    tma_store_2d_hint(map, slot, col, row0, l2_policy_evict_first());
    bulk_commit_group();
  }
}

// As drain64_release_to_global_act, the output leaving through the warp's staging slot
// and TMA stores (stage_store64) instead of stores from registers.
template <bool BF16, int ACT>
__device__ __noinline__ void drain64_release_to_staging_act(uint32_t tm_lane, uint32_t col0,
                                                            int ncols, uint32_t slot,
                                                            const CUtensorMap* map, int32_t row0,
                                                            int64_t rows, int lane,
                                                            uint32_t release) {
  const int head = ncols - 128;   // columns drained before the last 128
  for (int c = 0; c < head; c += 64) {
    uint32_t r[64], v[32];
    tmem_ld64x(tm_lane + col0 + c, r);
    tmem_wait_ld64(r);
    pack64<BF16, ACT>(r, v);
    stage_store64(v, slot, map, c, row0, rows, lane);
  }
  uint32_t r0[64], r1[64];
  tmem_ld64x(tm_lane + col0 + head, r0);
  tmem_ld64x(tm_lane + col0 + head + 64, r1);
  tmem_wait_ld64(r0);
  tmem_tie64(r1);
  tc_fence_before_sync();
  __syncwarp();
  if (lane == 0) mbar_arrive_remote(release);
  uint32_t v0[32], v1[32];
  pack64<BF16, ACT>(r0, v0);
  pack64<BF16, ACT>(r1, v1);
  stage_store64(v0, slot, map, head, row0, rows, lane);
  stage_store64(v1, slot, map, head + 64, row0, rows, lane);
}

template <bool BF16>
__device__ __forceinline__ void drain64_release_to_staging(int act, uint32_t tm_lane,
                                                           uint32_t col0, int ncols,
                                                           uint32_t slot, const CUtensorMap* map,
                                                           int32_t row0, int64_t rows, int lane,
                                                           uint32_t release) {
  if (act == 2)
    drain64_release_to_staging_act<BF16, 2>(tm_lane, col0, ncols, slot, map, row0, rows, lane,
                                            release);
  else if (act == 1)
    drain64_release_to_staging_act<BF16, 1>(tm_lane, col0, ncols, slot, map, row0, rows, lane,
                                            release);
  else
    drain64_release_to_staging_act<BF16, 0>(tm_lane, col0, ncols, slot, map, row0, rows, lane,
                                            release);
}

template <bool BF16>
__device__ __forceinline__ void drain64_release_to_global(int act, uint32_t tm_lane,
                                                          uint32_t col0, int ncols, uint8_t* out,
                                                          int64_t out_row0, int64_t rows, int ld,
                                                          int nvalid, int lane, uint32_t release) {
  if (act == 2)
    drain64_release_to_global_act<BF16, 2>(tm_lane, col0, ncols, out, out_row0, rows, ld, nvalid,
                                           lane, release);
  else if (act == 1)
    drain64_release_to_global_act<BF16, 1>(tm_lane, col0, ncols, out, out_row0, rows, ld, nvalid,
                                           lane, release);
  else
    drain64_release_to_global_act<BF16, 0>(tm_lane, col0, ncols, out, out_row0, rows, ld, nvalid,
                                           lane, release);
}

template <bool BF16>
__device__ __forceinline__ void drain64_to_global(int act, uint32_t tm_lane, uint32_t col0,
                                                  int ncols, uint8_t* out, int64_t out_row0,
                                                  int64_t rows, int ld, int nvalid, int lane) {
  if (act == 2)
    drain64_to_global_act<BF16, 2>(tm_lane, col0, ncols, out, out_row0, rows, ld, nvalid, lane);
  else if (act == 1)
    drain64_to_global_act<BF16, 1>(tm_lane, col0, ncols, out, out_row0, rows, ld, nvalid, lane);
  else
    drain64_to_global_act<BF16, 0>(tm_lane, col0, ncols, out, out_row0, rows, ld, nvalid, lane);
}

// Elementwise max of two packed fp16/bf16 pairs.
template <bool BF16>
__device__ __forceinline__ uint32_t max2(uint32_t a, uint32_t b) {
  uint32_t r;
  if constexpr (BF16)
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  else
    asm("max.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Pool epilogue.  Tile row = 16 * h + w over an 8 x 16 conv-output tile, so warp q holds
// conv rows 2q and 2q+1: the horizontal partner of a pixel sits in lane ^ 1 and the
// vertical one in lane ^ 16.  Each pixel's biased accumulators are rounded with ReLU to
// packed pairs first -- exactly the unfused operator's output -- and the 2x2 max is taken
// over those pairs (two shuffles and two packed maxes per pair of channels); the lane
// owning the window's top-left pixel stores the pooled pixel.
template <bool BF16>
__device__ __noinline__ void drain_pool(uint32_t tm_lane, uint32_t col0, int ncols,
                                        uint32_t tile, int q, int lane) {
  const bool owner = (lane & 17) == 0;
  const int prow = q * 8 + (lane >> 1);
  for (int c = 0; c < ncols; c += 32) {
    const bool two = c + 16 < ncols;
    uint32_t a[16], b[16], v[8], w[8];
    tmem_ld32(tm_lane + col0 + c, two, a, b);
    tmem_wait_ld(a, b);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[j] = pack2<BF16, true>(__uint_as_float(a[2 * j]), __uint_as_float(a[2 * j + 1]));
      w[j] = pack2<BF16, true>(__uint_as_float(b[2 * j]), __uint_as_float(b[2 * j + 1]));
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[j] = max2<BF16>(v[j], __shfl_xor_sync(0xffffffffu, v[j], 1));
      w[j] = max2<BF16>(w[j], __shfl_xor_sync(0xffffffffu, w[j], 1));
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[j] = max2<BF16>(v[j], __shfl_xor_sync(0xffffffffu, v[j], 16));
      w[j] = max2<BF16>(w[j], __shfl_xor_sync(0xffffffffu, w[j], 16));
    }
    if (owner) {
      st_row16_sw128(tile, prow, c, kPoolChunkBytes, v);
      if (two) st_row16_sw128(tile, prow, c + 16, kPoolChunkBytes, w);
    }
  }
}

template <bool A4D>
__device__ __forceinline__ void store_tile(const ChainParams& p, const CUtensorMap* tmOut,
                                           uint32_t tile, int nchunks, const TileCoord& tc) {
  if (!A4D && p.out_box3) {   // [N/64][M][64] view: the whole tile in one box
    tma_store_3d(tmOut, tile, 0, tc.m0, 0);
    return;
  }
  for (int nc = 0; nc < nchunks; ++nc) {
    if constexpr (A4D)
      tma_store_4d(tmOut, tile + nc * kPChunkBytes, nc * 64, tc.wo0, tc.ho0, tc.n);
    else
      tma_store_2d(tmOut, tile + nc * kPChunkBytes, nc * 64, tc.m0);
  }
}

// Warp-uniform bounded wait: every lane acquires the barrier itself, and the warp agrees
// on the outcome, so warp-collective tcgen05 loads and the named barriers below are
// always executed by whole warps.
__device__ __forceinline__ bool warp_wait(bool alive, uint32_t bar, uint32_t parity,
                                          const ChainParams& p, volatile uint32_t* abort_flag,
                                          uint32_t site, int32_t t) {
  bool ok = alive && mbar_wait(bar, parity, p.wait_limit_ns, abort_flag, p.err, p.kernel_id, site, t);
  return __all_sync(0xffffffffu, ok);
}

// Epilogue warps.  With epi_groups == 2 warpgroup g (warps 2+4g .. 5+4g) takes the
// CTA's tiles i with i & 1 == g and owns buffer g; with epi_groups == 1 all eight warps
// take every tile and warpgroup g drains the 32-column blocks 2k + g.
template <int MODE, bool A4D, bool BF16, bool WIDE, bool PAIR, bool NOPAIR, bool W0RES, bool TWO>
__device__ void epilogue_role(const ChainParams& p, const CUtensorMap* tmOut, uint32_t base,
                              uint32_t bars, uint32_t tmem_base,
                              volatile uint32_t* abort_flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wg = (warp - 2) >> 2;             // warpgroup 0 or 1
  const int q = warp & 3;                     // TMEM lane quadrant this warp may access
  const int row = q * 32 + lane;
  const uint32_t tm_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
  const int groups = PAIR ? 2 : p.epi_groups;   // tile pairs: alternate tiles
  const int g = groups == 2 ? wg : 0;         // which tiles
  const int c_first = groups == 2 ? 0 : 32 * wg;   // which columns
  const int c_step = groups == 2 ? 32 : 64;
  const uint32_t group_threads = static_cast<uint32_t>(kNumEpiThreads / groups);
  const uint32_t bar_id = 1u + static_cast<uint32_t>(g);
  const bool elected = threadIdx.x == 64 + g * static_cast<int>(group_threads);
  bool alive = true;
  Tracer trace(p, 2u + static_cast<uint32_t>(g), elected ? 1u : 0u);
  const uint32_t sb = groups == 2 ? static_cast<uint32_t>(g) : 0u;   // staging buffer
  const uint32_t out_tile = base + p.off_out[sb];

  // Chain, first half: GEMM0's accumulator -> P (shared memory or TMEM) -> P_FULL.
  auto epi0 = [&](int it) {
    const int32_t t = blockIdx.x + it * gridDim.x;
    const uint32_t b = buf_of(p, it), u = use_of(p, it);
    const uint32_t p_tile = base + p.off_p[b];
    alive = warp_wait(alive, bars + 8u * (BAR_ACC_FULL0 + b), u, p, abort_flag,
                      SITE_EPI_ACC_FULL, t);
    if (elected) trace(EV_EPI_ACC_READY, g, it);
    tc_fence_after_sync();
    if (!PAIR && p.out_alias_p) {   // P[b] doubles as this group's previous output staging
      if (elected) bulk_wait_read_all();
      named_bar_sync(bar_id, group_threads);
    }
    if (alive) {
      if (PAIR || (!NOPAIR && p.p_tmem))
        drain_to_tmem<BF16>(p.act0, tm_lane, p.d0_col[b], p.N0p, p.pt_col[b]);
      else
        drain_to_smem<BF16>(p.act0, tm_lane, p.d0_col[b], c_first, c_step, p.N0p, p_tile,
                            row, kPChunkBytes);
    }
    tc_fence_before_sync();
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8u * (BAR_P_FULL0 + b));
    if (elected) trace(EV_EPI_P_DONE, g, it);
  };

  // Chain, second half: GEMM1's accumulator -> output staging -> TMA store.
  auto epi1 = [&](int it) {
    const int32_t t = blockIdx.x + it * gridDim.x;
    const TileCoord tc = tile_coord<A4D>(p, t);
    const uint32_t b = buf_of(p, it), u = use_of(p, it);
    alive = warp_wait(alive, bars + 8u * (BAR_D1_FULL0 + b), u, p, abort_flag,
                      SITE_EPI_D1_FULL, t);
    if (elected) trace(EV_EPI_D1_READY, g, it);
    tc_fence_after_sync();
    if constexpr (W0RES) {
      // Straight from registers to the output rows (no staging tile, no TMA store); then
      // the buffer (D0 -> P + D1) may take tile i + 2.
      const int32_t m = tc.m0 + row;
      if (alive)   // warp-uniform: the drain's TMEM loads are warp-collective
        drain_to_global<BF16>(p.act1, tm_lane, p.d1_col[b], p.N1p,
                              p.out_ptr + static_cast<size_t>(m < p.M ? m : 0) *
                                              static_cast<size_t>(p.out_ld) * 2u,
                              p.N1, m < p.M);
      if (elected) trace(EV_EPI_DRAINED, g, it);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + 8u * (BAR_ACC_EMPTY0 + b));
      if (elected) trace(EV_EPI_STORED, g, it);
      return;
    }
    if constexpr (TWO && A4D) {
      // (out_slots) Row 32q + lane of the 8 x 16 tile is pixel (ho0 + 2q + lane / 16,
      // wo0 + lane % 16): each warp stores its two output rows from its own slot.  Nothing
      // waits for this buffer's D1 but GEMM1 of the group's next tile, which follows the
      // group's next P.
      const int32_t h0 = tc.ho0 + 2 * q;
      const uint32_t slot =
          base + p.off_out[0] + static_cast<uint32_t>(warp - 2) * kOutSlotBytes;
      if (alive)   // warp-uniform: the drain's TMEM loads are warp-collective
        drain16_to_slot<BF16>(p.act1, tm_lane, p.d1_col[b], p.N1p, p.N1, slot, tmOut, tc.wo0,
                              h0, tc.n, h0 < p.Ho && !*abort_flag, lane);
      tc_fence_before_sync();
      if (elected) trace(EV_EPI_STORED, g, it);
      return;
    }
    if (PAIR || !p.out_alias_p) {
      if (elected) bulk_wait_read_all();
      named_bar_sync(bar_id, group_threads);
    }
    if (elected) trace(EV_EPI_STAGING, g, it);
    if (alive)
      drain_to_smem<BF16>(p.act1, tm_lane, p.d1_col[b], c_first, c_step, p.N1p, out_tile,
                          row, kPChunkBytes);
    if (elected) trace(EV_EPI_DRAINED, g, it);
    tc_fence_before_sync();
    if (PAIR || (!NOPAIR && p.p_tmem)) {   // the buffer (D0 -> P + D1) may take tile i + 2
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + 8u * (BAR_ACC_EMPTY0 + b));
    }
    fence_proxy_async_smem();
    named_bar_sync(bar_id, group_threads);
    if (elected && !*abort_flag) {
      store_tile<A4D>(p, tmOut, out_tile, (p.N1p + 63) >> 6, tc);
      bulk_commit_group();
      trace(EV_EPI_STORED, g, it);
    }
  };

  // Three-operator chain, middle: GEMM1's accumulator -> P1 (shared memory) -> P1_FULL.
  auto epi1_p1 = [&](int it) {
    const int32_t t = blockIdx.x + it * gridDim.x;
    const uint32_t b = buf_of(p, it), u = use_of(p, it);
    alive = warp_wait(alive, bars + 8u * (BAR_D1_FULL0 + b), u, p, abort_flag,
                      SITE_EPI_D1_FULL, t);
    if (elected) trace(EV_EPI_D1_READY, g, it);
    tc_fence_after_sync();
    if (alive)
      drain_to_smem<BF16>(p.act1, tm_lane, p.d1_col[b], c_first, c_step, p.N1p,
                          base + p.off_p1[b], row, kPChunkBytes);
    tc_fence_before_sync();
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8u * (BAR_P1_FULL0 + b));
    if (elected) trace(EV_EPI_P1_DONE, g, it);
  };

  // Three-operator chain, last: GEMM2's accumulator -> output staging -> TMA store.
  auto epi2 = [&](int it) {
    const int32_t t = blockIdx.x + it * gridDim.x;
    const TileCoord tc = tile_coord<A4D>(p, t);
    const uint32_t b = buf_of(p, it), u = use_of(p, it);
    alive = warp_wait(alive, bars + 8u * (BAR_D2_FULL0 + b), u, p, abort_flag,
                      SITE_EPI_D2_FULL, t);
    tc_fence_after_sync();
    if (elected) bulk_wait_read_all();   // this group's staging is free again
    named_bar_sync(bar_id, group_threads);
    if (elected) trace(EV_EPI_STAGING, g, it);
    if (alive)
      drain_to_smem<BF16>(p.act2, tm_lane, p.d2_col[b], c_first, c_step, p.N2p, out_tile, row,
                          kPChunkBytes);
    tc_fence_before_sync();
    fence_proxy_async_smem();
    named_bar_sync(bar_id, group_threads);
    if (elected && !*abort_flag) {
      store_tile<A4D>(p, tmOut, out_tile, (p.N2p + 63) >> 6, tc);
      bulk_commit_group();
      trace(EV_EPI_STORED, g, it);
    }
  };

  const int ntiles = local_tiles(p);
  if constexpr (MODE == MODE_CHAIN && WIDE) {
    // Wide chains (one group of both warpgroups): warpgroup wg packs half wg of D0 into P
    // in place and publishes it on P_FULL[wg] (four warps); then both drain D1, 32 of every
    // 64 columns each, and free the tile's TMEM on ACC_EMPTY[0] (eight warps).  Every
    // barrier completes once per tile, so tile it waits on parity it & 1.
    for (int it = 0; it < ntiles; ++it) {
      const int32_t t = blockIdx.x + it * gridDim.x;
      const uint32_t u = static_cast<uint32_t>(it) & 1u;
      alive = warp_wait(alive, bars + 8u * (BAR_ACC_FULL0 + wg), u, p, abort_flag,
                        SITE_EPI_ACC_FULL, t);
      if (elected) trace(EV_EPI_ACC_READY, wg, it);
      tc_fence_after_sync();
      const int c0 = 256 * wg, n = min(256, p.N0p - c0);
      if (alive && n > 0)
        drain_to_tmem<BF16>(p.act0, tm_lane, static_cast<uint32_t>(c0), n,
                            static_cast<uint32_t>(c0));
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + 8u * (BAR_P_FULL0 + wg));
      if (elected) trace(EV_EPI_P_DONE, wg, it);

      const TileCoord tc = tile_coord<A4D>(p, t);
      alive = warp_wait(alive, bars + 8u * BAR_D1_FULL0, u, p, abort_flag, SITE_EPI_D1_FULL, t);
      if (elected) trace(EV_EPI_D1_READY, 0, it);
      tc_fence_after_sync();
      if (elected) bulk_wait_read_all();   // the staging is free again
      named_bar_sync(bar_id, group_threads);
      if (elected) trace(EV_EPI_STAGING, 0, it);
      if (alive)
        drain_to_smem<BF16>(p.act1, tm_lane, p.d1_col[it & 1], c_first, c_step, p.N1p, out_tile,
                            row, kPChunkBytes);
      if (elected) trace(EV_EPI_DRAINED, 0, it);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + 8u * BAR_ACC_EMPTY0);
      fence_proxy_async_smem();
      named_bar_sync(bar_id, group_threads);
      if (elected && !*abort_flag) {
        store_tile<A4D>(p, tmOut, out_tile, (p.N1p + 63) >> 6, tc);
        bulk_commit_group();
        trace(EV_EPI_STORED, 0, it);
      }
    }
  } else if (MODE == MODE_CHAIN3) {
    for (int it = g; it < ntiles; it += groups) {
      epi0(it);
      epi1_p1(it);
      epi2(it);
    }
  } else if (MODE == MODE_CHAIN && !PAIR && p.nbuf_log2 == 2) {
    // Four buffers: the group runs the first half of its next tile before the second half
    // of the current one, so that it drains GEMM0 while GEMM1 of the current tile runs.
    if (g < ntiles) epi0(g);
    for (int it = g; it < ntiles; it += groups) {
      if (it + groups < ntiles) epi0(it + groups);
      epi1(it);
    }
  } else if (MODE == MODE_CHAIN) {
    for (int it = g; it < ntiles; it += groups) {
      epi0(it);
      epi1(it);
    }
  } else {
    for (int it = g; it < ntiles; it += groups) {
      const int32_t t = blockIdx.x + it * gridDim.x;
      const TileCoord tc = tile_coord<A4D>(p, t);
      const uint32_t b = buf_of(p, it), u = use_of(p, it);
      alive = warp_wait(alive, bars + 8u * (BAR_ACC_FULL0 + b), u, p, abort_flag,
                        SITE_EPI_ACC_FULL, t);
      if (elected) trace(EV_EPI_ACC_READY, g, it);
      tc_fence_after_sync();
      if (elected) bulk_wait_read_all();   // this group's staging is free again
      named_bar_sync(bar_id, group_threads);
      if (elected) trace(EV_EPI_STAGING, g, it);
      if (alive) {
        if (MODE == MODE_POOL)
          drain_pool<BF16>(tm_lane, p.d0_col[b], p.N0p, out_tile, q, lane);
        else
          drain_to_smem<BF16>(p.act0, tm_lane, p.d0_col[b], c_first, c_step, p.N0p, out_tile,
                              row, kPChunkBytes);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + 8u * (BAR_ACC_EMPTY0 + b));
      fence_proxy_async_smem();
      named_bar_sync(bar_id, group_threads);
      if (elected && !*abort_flag) {
        if (MODE == MODE_POOL) {
          const int nch = (p.N0p + 63) >> 6;
          for (int nc = 0; nc < nch; ++nc)
            tma_store_4d(tmOut, out_tile + nc * kPoolChunkBytes, nc * 64, tc.wo0 >> 1,
                         tc.ho0 >> 1, tc.n);
        } else {
          store_tile<A4D>(p, tmOut, out_tile, (p.N0p + 63) >> 6, tc);
        }
        bulk_commit_group();
        trace(EV_EPI_STORED, g, it);
      }
    }
  }
  // The staging tiles must outlive the stores' reads of them; the writes themselves are
  // complete when the grid is.  (Two-issuer chain: lane 0 of every warp stored.)
  if (TWO ? lane == 0 : elected) bulk_wait_read_all();
}

// ------------------------------------------------------------------------------------
// bias operands
// ------------------------------------------------------------------------------------
// The bias enters every GEMM as one more K step after the last chunk, D += ONES . BIAS, so
// the epilogue never reads it.  ONES is a K-major 128B-swizzled A tile whose row m holds 1 at
// k = 0 and 0 at k = 1..15; all its 8-row groups are equal, so the descriptor's group
// stride is 0 and the tile is a single 1 KiB swizzle atom (row r, k = 0 sits at byte
// r * 128 + (0 ^ r) * 16).  BIAS is an MN-major 128B-swizzled B tile with 16 k-rows per
// 64-wide N block (2 KiB): k-row 0 holds the block's 64 biases (unswizzled, as row 0),
// the other rows are 0.  The product is the bias broadcast to all 128 rows, exact in
// fp32.  Written by the epilogue warps with generic stores.
template <bool BF16>
__device__ __forceinline__ void fill_bias_operands(const ChainParams& p, uint8_t* region,
                                                   int tid, int nthreads, int ngemms) {
  const int n0blk = (p.N0p + 63) >> 6;
  const int n1blk = ngemms >= 2 ? (p.N1p + 63) >> 6 : 0;
  const int n2blk = ngemms >= 3 ? (p.N2p + 63) >> 6 : 0;
  // Each thread fetches its first element of every bias row before the fill below, so the
  // global loads overlap it instead of following one another (rows longer than nthreads,
  // N0 up to 512, finish in the loop at the end).
  const uint16_t v0 = (tid < p.N0 && p.b0 != nullptr) ? p.b0[tid] : uint16_t(0);
  const uint16_t v1 = (ngemms >= 2 && tid < p.N1 && p.b1 != nullptr) ? p.b1[tid] : uint16_t(0);
  const uint16_t v2 = (ngemms >= 3 && tid < p.N2 && p.b2 != nullptr) ? p.b2[tid] : uint16_t(0);
  // ONES, and every byte of the BIAS blocks but their k-row 0 (bytes [0, 128) of a block).
  uint32_t* words = reinterpret_cast<uint32_t*>(region);
  const int nwords = (static_cast<int>(kOnesBytes) +
                      (n0blk + n1blk + n2blk) * static_cast<int>(kBiasBlockBytes)) >> 2;
  const uint32_t one = BF16 ? 0x3F80u : 0x3C00u;
  for (int w = tid; w < nwords; w += nthreads) {
    const int o = w << 2;
    if (o < static_cast<int>(kOnesBytes))
      words[w] = o == (o >> 7) * 144 ? one : 0u;   // row r: byte r * 128 + r * 16
    else if (((o - static_cast<int>(kOnesBytes)) & static_cast<int>(kBiasBlockBytes - 1)) >= 128)
      words[w] = 0u;
  }
  // k-row 0 of block n / 64 holds element n at byte 2 * (n % 64); zero beyond N.
  uint16_t* halves = reinterpret_cast<uint16_t*>(region + kOnesBytes);
  constexpr int kBlockHalves = static_cast<int>(kBiasBlockBytes / 2);
  if (tid < n0blk * 64) halves[(tid >> 6) * kBlockHalves + (tid & 63)] = v0;
  if (tid < n1blk * 64) halves[(n0blk + (tid >> 6)) * kBlockHalves + (tid & 63)] = v1;
  if (tid < n2blk * 64) halves[(n0blk + n1blk + (tid >> 6)) * kBlockHalves + (tid & 63)] = v2;
  for (int n = tid + nthreads; n < n0blk * 64; n += nthreads)   // wide N0
    halves[(n >> 6) * kBlockHalves + (n & 63)] =
        (n < p.N0 && p.b0 != nullptr) ? p.b0[n] : uint16_t(0);
}

// W2 [N1][N2] (row-major, global) -> the resident MN-major layout GEMM2 reads, as a TMA
// load with 128-byte swizzle would lay it out: per 64-row K chunk kc and 64-wide N block
// nb an 8 KiB block, K-row r at r * 128 bytes, its 16-byte unit j (columns 8j..8j+7) at
// unit j ^ (r % 8); rows beyond N1 and columns beyond N2 are zero.  Generic stores by the
// epilogue warps, before they release the bias operands (the MMA issuer waits for those
// before the first MMA that could read W2).
__device__ __forceinline__ void fill_w2(const ChainParams& p, uint8_t* dst, int tid,
                                        int nthreads) {
  const int nblk = (p.N2p + 63) >> 6;
  const int units = p.kchunks2 * nblk * 64 * 8;   // 16-byte units
  for (int u = tid; u < units; u += nthreads) {
    const int j = u & 7, r = (u >> 3) & 63, blk = u >> 9;
    const int nb = blk % nblk, kc = blk / nblk;
    const int k = kc * 64 + r, n = nb * 64 + j * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (k < p.N1 && n < p.N2)
      v = *reinterpret_cast<const uint4*>(p.w2 + static_cast<size_t>(k) * p.N2 + n);
    *reinterpret_cast<uint4*>(dst + static_cast<size_t>(kc) * p.w2_chunk_bytes + nb * 8192 +
                              r * 128 + ((j ^ (r & 7)) << 4)) = v;
  }
}

// ------------------------------------------------------------------------------------
// the kernel
// ------------------------------------------------------------------------------------
template <int MODE, bool A4D, bool W0MN, bool W1MN, bool BF16, bool WIDE = false,
          bool PAIR = false, bool NOPAIR = false, bool W0RES = false, bool TWO = false>
__global__ void __launch_bounds__(chain_threads(MODE, TWO), 1)
    chain_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW0,
                 const __grid_constant__ CUtensorMap tmW1,
                 const __grid_constant__ CUtensorMap tmOut, const ChainParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t bars = base + p.off_bar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + p.off_bar + 8u * BAR_COUNT);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t warps_per_group = static_cast<uint32_t>(kNumEpiWarps / p.epi_groups);
  Tracer ktrace(p, 1, threadIdx.x == 32 ? 1u : 0u);
  ktrace(EV_KERNEL_ENTRY, 0, 0);
  // Each launch's parameter block starts cold in the constant cache, and every role's
  // first reads of it would miss one line after another.  One word of each 64-byte line is
  // read here by a thread of its own, all at once, while the previous grid may still run.
  constexpr uint32_t kParamLines = (sizeof(ChainParams) + 63u) / 64u;
  if (threadIdx.x >= 64u && threadIdx.x < 64u + kParamLines) {
    const uint32_t w = reinterpret_cast<const uint32_t*>(&p)[(threadIdx.x - 64u) * 16u];
    asm volatile("" ::"r"(w));
  }

  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < p.num_stages; ++s) {
      mbar_init(bars + 8u * (BAR_FULL0 + s), 1);
      mbar_init(bars + 8u * (BAR_EMPTY0 + s), 1);
    }
    mbar_init(bars + 8u * BAR_WFULL, 1);
    for (uint32_t a = 0; a < kMaxBufs; ++a) {
      mbar_init(bars + 8u * (BAR_ACC_FULL0 + a), 1);
      mbar_init(bars + 8u * (BAR_ACC_EMPTY0 + a), warps_per_group);
      mbar_init(bars + 8u * (BAR_P_FULL0 + a), WIDE ? 4u : warps_per_group);
      mbar_init(bars + 8u * (BAR_D1_FULL0 + a), 1);
      if (MODE == MODE_CHAIN3) {
        mbar_init(bars + 8u * (BAR_P1_FULL0 + a), warps_per_group);
        mbar_init(bars + 8u * (BAR_D2_FULL0 + a), 1);
      }
    }
    mbar_init(bars + 8u * BAR_MMA_DONE, two_issuers(MODE, TWO) && p.two_issuers ? 2u : 1u);
    mbar_init(bars + 8u * BAR_BIAS_READY, kNumEpiWarps);
    if (W0RES)
      for (uint32_t c = 0; c < static_cast<uint32_t>(kMaxW0Chunks); ++c)
        mbar_init(bars + 8u * (BAR_W0C0 + c), 1);
    *abort_flag = 0u;
    fence_barrier_init();
    fence_proxy_async_smem();
    // Once every CTA of this grid has passed this point, the next kernel may be
    // scheduled; its CTAs take an SM as this grid's CTAs leave and wait for this grid
    // before touching global memory.
    grid_launch_dependents();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmW0);
    if (MODE == MODE_CHAIN || MODE == MODE_CHAIN3) tma_prefetch_desc(&tmW1);
    tma_prefetch_desc(&tmOut);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  ktrace(EV_SETUP_DONE, 0, 0);

  // Loads and stores of global memory wait for the previous kernel of the stream to
  // complete (inputs may be its outputs, outputs its inputs): every role executes
  // griddepcontrol.wait before its first one.  The L2 prefetches just below are issued
  // BEFORE that wait.  They are hints that move no data into the CTA and write nothing:
  // a line the previous kernel is still writing is kept coherent in L2 (the point where
  // its stores land), so a prefetch at worst warms a line that is rewritten later, and
  // the TMA loads issued after the wait read the final data.
  if (warp == 0) {
    // The first tile's A (and, if the plan asks, the second's) and (from one CTA) the
    // weights into L2 while the previous kernel finishes.
    if (lane == 0) {
      prefetch_a_tile(p, blockIdx.x);
      if (p.pf_second) prefetch_a_tile(p, blockIdx.x + gridDim.x);
      if (blockIdx.x == 0) {
        bulk_prefetch_l2(p.pf_w0, p.pf_w0_bytes);
        if (MODE == MODE_CHAIN || MODE == MODE_CHAIN3) bulk_prefetch_l2(p.pf_w1, p.pf_w1_bytes);
      }
    }
    __syncwarp();
    producer_role<MODE, A4D, W0MN, W1MN, WIDE, PAIR, NOPAIR, W0RES, TWO>(p, &tmA, &tmW0, &tmW1, base,
                                                                   bars, abort_flag);
    __syncwarp();
  } else if (warp == 1) {
    mma_role<MODE, A4D, W0MN, W1MN, BF16, WIDE, PAIR, NOPAIR, W0RES, TWO>(p, base, bars, tmem_base,
                                                                    abort_flag, 0);
    __syncwarp();
  } else if (two_issuers(MODE, TWO) && warp == kSecondIssuerWarp) {
    if (p.two_issuers)
      mma_role<MODE, A4D, W0MN, W1MN, BF16, WIDE, PAIR, NOPAIR, W0RES, TWO>(p, base, bars, tmem_base,
                                                                      abort_flag, 1);
    __syncwarp();
  } else {
    // The bias operands, off the producer's critical path; the MMA issuer waits for them
    // before its first MMA.
    grid_dependency_wait();
    fill_bias_operands<BF16>(p, base_ptr + p.off_bias, static_cast<int>(threadIdx.x) - 64,
                             kNumEpiThreads,
                             MODE == MODE_CHAIN3 ? 3 : (MODE == MODE_CHAIN ? 2 : 1));
    if (MODE == MODE_CHAIN3)
      fill_w2(p, base_ptr + p.off_w2, static_cast<int>(threadIdx.x) - 64, kNumEpiThreads);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8u * BAR_BIAS_READY);
    epilogue_role<MODE, A4D, BF16, WIDE, PAIR, NOPAIR, W0RES, TWO>(p, &tmOut, base, bars, tmem_base,
                                                              abort_flag);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

}  // namespace B2B_KNS
}  // namespace b2b
