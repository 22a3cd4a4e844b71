// kernel_params.h -- launch parameters shared by the host planner and the chain kernel.
#pragma once

#include <cstdint>

namespace b2b {

// What one launch of the chain kernel computes.
enum ChainMode : int {
  MODE_CHAIN = 0,   // GEMM0 -> epilogue0 -> P (smem) -> GEMM1 -> epilogue1 -> global
  MODE_SINGLE = 1,  // GEMM0 -> epilogue0 -> global (one operator of the unfused path)
  MODE_POOL = 2,    // GEMM0 (conv) -> 2x2 max -> bias -> ReLU -> global (pooled)
  MODE_CHAIN3 = 3,  // GEMM0 -> P0 (smem) -> GEMM1 -> P1 (smem) -> GEMM2 -> global
};

// Kernel ids recorded in the device error word.
enum KernelId : uint32_t {
  KID_GEMM_CHAIN = 1,
  KID_CONV1X1_CHAIN = 2,
  KID_CONV_CHAIN = 3,
  KID_GEMM_SINGLE = 4,
  KID_CONV1X1_SINGLE = 5,
  KID_CONV_SINGLE = 6,
  KID_CONV_POOL = 7,
  KID_GEMM_CHAIN3 = 8,
  KID_GEMM_CHAIN_CTA2 = 9,   // b2b GEMM chain over CTA pairs (cta_group::2)
  KID_CONV_POOL_CTA2 = 10,   // conv + pool over CTA pairs
  KID_PROBE = 15,
};

// Wait sites recorded in the device error word.
enum WaitSite : uint32_t {
  SITE_PRODUCER_EMPTY = 1,
  SITE_MMA_WEIGHTS = 2,
  SITE_MMA_FULL = 3,
  SITE_MMA_ACC_EMPTY = 4,
  SITE_MMA_P_FULL = 5,
  SITE_MMA_DRAIN = 6,
  SITE_EPI_ACC_FULL = 7,
  SITE_EPI_D1_FULL = 8,
  SITE_PRODUCER_DRAIN = 9,
  SITE_PROBE = 10,
  SITE_MMA_P1_FULL = 11,
  SITE_EPI_D2_FULL = 12,
};

// Events of the optional trace: one CTA's roles stamp clock64() at these points.
enum TraceEvent : uint32_t {
  EV_PROD_ACQUIRE = 1,   // producer got a free ring slot
  EV_PROD_ISSUED = 2,    // producer issued the slot's TMA loads
  EV_MMA_FULL = 3,       // MMA issuer saw a ring slot filled
  EV_MMA_G0_DONE = 4,    // GEMM0 of a tile issued and committed
  EV_MMA_P_READY = 5,    // MMA issuer saw a P tile published
  EV_MMA_G1_DONE = 6,    // GEMM1 of a tile issued and committed
  EV_MMA_ACC_FREE = 7,   // MMA issuer saw an accumulator drained (single/pool)
  EV_EPI_ACC_READY = 8,  // epilogue group saw GEMM0's accumulator complete
  EV_EPI_P_DONE = 9,     // epilogue group published P
  EV_EPI_D1_READY = 10,  // epilogue group saw GEMM1's accumulator complete
  EV_EPI_STAGING = 11,   // epilogue group's output staging free
  EV_EPI_STORED = 12,    // epilogue group issued the tile's TMA store
  EV_MMA_WAIT = 13,      // MMA issuer starts waiting for a ring slot
  EV_MMA_ISSUED = 14,    // MMA issuer issued a slot's MMAs
  EV_PROD_W1_ISSUED = 15,  // producer issued a streamed GEMM1 weight chunk
  EV_MMA_W1_FULL = 16,     // MMA issuer saw a streamed GEMM1 weight chunk land
  EV_KERNEL_ENTRY = 17,    // first instruction of the CTA
  EV_EPI_DRAINED = 18,     // epilogue group's elected thread finished its output drain
  EV_SETUP_DONE = 19,      // barriers initialised and TMEM allocated (after __syncthreads)
  EV_DEP_READY = 20,       // the MMA warp's wait for the previous grid returned
  EV_EPI_P1_DONE = 21,     // three-operator chain: epilogue group published P1
  EV_MMA_G2_DONE = 22,     // three-operator chain: GEMM2 of a tile issued and committed
  EV_PROD_START = 23,      // producer past its wait for the previous grid
  EV_MMA_SETUP = 24,       // MMA issuer's descriptors ready, before its first wait
};

constexpr int kBlockM = 128;          // rows of one tile = TMEM lanes = tcgen05 M
constexpr int kChunkK = 64;           // K elements per staged chunk (128 B rows, SW128)
constexpr int kNumEpiWarps = 8;       // two warpgroups of four (one per TMEM lane quadrant)
constexpr int kNumEpiThreads = 32 * kNumEpiWarps;
constexpr int kNumThreads = 64 + kNumEpiThreads;   // warp 0 TMA, warp 1 MMA + TMEM, 2..9 epilogue
// The conv + pool kernel (MODE_POOL) and the conv chain's two-issuer instantiation (the
// kernel's TWO template parameter, `two` below) add warp 10, a possible second MMA issuer
// (ChainParams::two_issuers): warps 1 and 10 then take alternate tiles (each its own
// accumulators), so that one issues while the other waits between ring stages or for its
// epilogue.  With N = 64 the tensor core finishes an MMA in ~48 cycles and accepts only a
// short queue of them, so every cycle a single issuer spends on barriers and bookkeeping
// leaves it idle.
__host__ __device__ constexpr bool two_issuers(int mode, bool two) {
  return mode == 2 || (mode == 0 && two);
}
__host__ __device__ constexpr int chain_threads(int mode, bool two) {
  return kNumThreads + (two_issuers(mode, two) ? 32 : 0);
}
constexpr int kSecondIssuerWarp = kNumThreads / 32;
constexpr int kMaxStages = 8;
constexpr int kMaxBufs = 4;          // accumulator / P buffers per CTA
// The conv + pool kernel over CTA pairs: up to three MMA issuers (warps 1, 10 and 11),
// each with two of up to six accumulators, over up to ten ring stages.
constexpr int kPool2MaxStages = 10;
constexpr int kPool2MaxBufs = 6;
constexpr int kThirdIssuerWarp = kSecondIssuerWarp + 1;
constexpr int kMaxW0Chunks = 8;      // K chunks of a W0 kept resident beside streamed W1
// Bias operands in shared memory (at off_bias): a 1 KiB ONES tile, then per GEMM one
// 2 KiB BIAS block per 64-wide N block.
constexpr uint32_t kOutSlotBytes = 1024;   // out_slots: 32 rows x 16 columns per warp
constexpr uint32_t kOnesBytes = 1024;
constexpr uint32_t kBiasBlockBytes = 2048;
constexpr uint32_t kABytes = kBlockM * kChunkK * 2;   // 16 KiB A chunk
constexpr uint32_t kPChunkBytes = kBlockM * 128;      // 128 rows x 64 cols x 2 B
constexpr uint32_t kPoolChunkBytes = 32 * 128;        // 4h x 8w pooled pixels x 64 ch

struct ChainParams {
  // --- problem -------------------------------------------------------------------
  int32_t M;            // rows (2D A) -- unused for conv tiles
  int32_t K0;           // GEMM0 reduction length (2D A) or input channels C (4D A)
  int32_t N0, N1;       // true output widths of GEMM0 / GEMM1
  int32_t N0p, N1p;     // padded to multiples of 16 (tcgen05 N granularity for M = 128)
  int32_t kchunks0;     // 64-wide K chunks of GEMM0 (4D: taps * kc_per_tap)
  int32_t kc_per_tap;   // 4D: ceil(C / 64)
  int32_t halo;         // 4D, resident filters, R > 1: one box of (8 + R - 1) x 16 pixels per
                        //   (column tap s, channel block) serves the R row taps
  int32_t kstages0;     // ring stages per tile for GEMM0 (halo: S * kc_per_tap; else kchunks0)
  uint32_t a_stage_bytes;   // A bytes per ring stage (16 KiB; halo: (8 + R - 1) * 2 KiB)
  int32_t kchunks1;     // 64-wide K chunks of GEMM1 (= ceil(N0p / 64))
  int32_t R, S, pad;    // 4D filter
  int32_t stride;       // 4D: spatial stride of the first conv (halo loads only at 1)
  int32_t Ho, Wo;       // 4D output spatial size (before pooling)
  int32_t tiles_w, tiles_h;  // 4D tiling: 16 output columns x 8 output rows per tile
  int32_t num_tiles;
  int32_t is_bf16;
  int32_t act0, act1;
  const uint16_t* b0;   // may be null
  const uint16_t* b1;   // may be null
  // --- three-operator chain (MODE_CHAIN3): GEMM2 over P1 = act1(D1) ------------------
  int32_t N2, N2p;      // GEMM2 output width, padded to 16
  int32_t kchunks2;     // 64-wide K chunks of GEMM2 (= ceil(N1p / 64))
  int32_t act2;
  const uint16_t* b2;   // may be null
  const uint16_t* w2;   // W2 [N1][N2] row-major in global memory; the epilogue warps copy
                        //    it into the swizzled resident layout at off_w2
  uint32_t w2_chunk_bytes, off_w2;
  uint32_t off_p1[2];   // P1 buffers (K-major, swizzled like P)
  uint32_t d2_col[2];   // TMEM columns of the GEMM2 accumulators
  // L2 prefetch (warming only): 2-D A (null for the implicit-GEMM conv A) with the bytes of
  // one 128-row tile and of the whole tensor, and the weights' bytes.
  const uint8_t* pf_a;
  uint64_t pf_a_bytes;
  uint32_t pf_a_tile_bytes;
  int32_t pf_second;    // 1: the CTA's second tile's A rows too, at the start
  const uint8_t* pf_w0;
  const uint8_t* pf_w1;
  uint32_t pf_w0_bytes, pf_w1_bytes;
  // --- shared-memory plan (byte offsets from the 1024-aligned dynamic base) -----------
  uint32_t off_ring, stage_bytes, num_stages;
  uint32_t w0_chunk_bytes, w1_chunk_bytes;
  uint32_t off_w0, off_w1;      // resident weights (resident != 0)
  uint32_t off_p[kMaxBufs], off_out[2], off_bias, off_bar;
  int32_t resident;             // 1: W0/W1 loaded once per CTA; 0: streamed per tile
  int32_t out_alias_p;          // 1: output staging b shares P buffer b
  int32_t nbuf_log2;            // log2 of the accumulator (and, chained, P) buffers: tile i
                                //    of the CTA uses buffer i mod 2^nbuf_log2 (4 buffers:
                                //    narrow smem-P chains, each epilogue group one tile ahead)
  int32_t acc_dual;             // 1: accumulators (and, chained, P) double-buffered:
                                //    tile i uses buffer i & 1, two tiles in flight
  int32_t p_tmem;               // 1 (chain): P is written back into TMEM over the consumed
                                //    GEMM0 columns and GEMM1 reads A from TMEM; tiles are
                                //    processed in pairs, buffer b holds D0 -> P + D1
  int32_t w0_box3, w1_box3;     // 1: a row-major weight (N a multiple of 64) is mapped as
                                //    [N/64][K][64], so one 3-D box loads a whole K chunk
  int32_t out_box3;             // 1: the 2-D output (N a multiple of 64) is mapped the same
                                //    way and a tile is stored by one 3-D box
  int32_t w0_res;               // 1 (P in TMEM, tile pairs): W0 alone is resident, loaded
                                //    once per CTA with one barrier per K chunk; A and W1
                                //    stream through the ring, and epilogue 1 stores the
                                //    output tile from registers straight to global memory
                                //    (no staging tile: W0 takes its shared memory)
  int32_t cta_pair;             // 1: the chain runs over CTA pairs (chain_cta2_kernel.cuh,
                                //    clusters of two CTAs, tcgen05 .cta_group::2); num_tiles
                                //    then counts 256-row tiles, and each CTA holds half of
                                //    W0 and of W1 (w0/w1_chunk_bytes are the halves' chunks)
  uint8_t* out_ptr;             // w0_res, cta_pair: the output D [M][out_ld] row-major
  int32_t out_ld;               // w0_res, cta_pair: elements per output row
  int32_t two_issuers;          // (MODE_POOL; MODE_CHAIN with 4-D A, resident filters and
                                //    P in TMEM) 1: warps 1 and 10 issue the MMAs of
                                //    alternate tiles, the ring split into two sub-rings
                                //    (subring_of); 0: warp 1 alone, warp 10 idle.  A chain
                                //    then keeps D1 apart from D0 / P in TMEM (buffer b =
                                //    issuer b) and stores its output with out_slots; the conv
                                //    + pool kernel over CTA pairs: the issuers beyond warp 1
                                //    (0, 1 or 2: warps 10 and 11), each with its own
                                //    sub-ring
  int32_t out_slots;            // (two-issuer conv chain) 1: each epilogue warp stages its 32
                                //    rows' output 16 columns at a time in a 1 KiB slot of
                                //    its own (kOutSlotBytes from off_out[0], unswizzled) and
                                //    stores it with TMA (box of 16 channels x 16 x 2 pixels)
  int32_t out_stage;            // cta_pair: 1 if each epilogue warp stages its 32 rows' output
                                //    64 columns at a time (4 KiB per warp from off_out[0],
                                //    128B-swizzled) and stores them with TMA; 0: stored
                                //    from registers
  int32_t w1_group;             // 1 (P in TMEM, streamed weights): W1 is loaded once per
                                //    pair of tiles, w1_per_stage chunks per ring stage,
                                //    and both tiles' GEMM1 read it from the same stages
  uint32_t w1_per_stage;        // W1 chunks per ring stage when w1_group
  uint32_t p_hi;                // (wide) TMEM column of the upper half's D0 and P
  uint32_t p_split;             // wide chains (256 < N0p <= 512, P in TMEM): 256, the
                                //    width of GEMM0's lower pass; GEMM0 runs in two passes
                                //    over the halves of N0 into TMEM columns [0, 256) and
                                //    [256, N0p), each half's P packed in place by one
                                //    warpgroup.  0 otherwise.
  int32_t epi_groups;           // 2: the epilogue warpgroups take alternate tiles;
                                // 1: both warpgroups split the columns of every tile
  uint32_t tmem_cols;
  uint32_t d0_col[kMaxBufs], d1_col[kMaxBufs];  // TMEM columns of the accumulator buffers
  uint32_t pt_col[2];           // (P in TMEM) TMEM column of buffer b's packed P: over its D0
                                //    (d0_col[b]), or, with two issuers, a region of its own
  uint64_t wait_limit_ns;
  uint32_t kernel_id;
  uint32_t* err;                // device error word {code, kernel, site, tile}
  unsigned long long* trace;    // optional event trace (see TraceEvent), or null
  uint32_t trace_cap;           // capacity of `trace` in events
  uint32_t trace_cta;           // the CTA whose events are recorded
};

}  // namespace b2b
