// chain_cta2_kernel.cuh -- the b2b GEMM chain over CTA pairs (tcgen05 .cta_group::2).
//
// Two CTAs on two SMs form a cluster and share every MMA: one tcgen05.mma of M = 256 rows
// takes rows 0..127 of A from the first CTA's shared memory and rows 128..255 from the
// second's, and columns [0, N/2) of B from the first CTA, [N/2, N) from the second; each
// CTA's TMEM receives its own 128 rows of D with all N columns.  For the chain this means
// each SM holds only HALF of W0 and half of W1, so both weights stay resident (W0 and W1
// of an FFN-like 256 -> 256 -> 128 chain take 96 KiB per SM instead of 192), every A chunk
// streams through a deep ring, and each SM reads half of B per MMA from shared memory.
// The chain is the same as the tile-pair schedule of chain_kernel.cuh (BOLT notes,
// "Persistent kernel (GEMM/Conv) fusion" and "Threadblock residence": the CTA pair owns
// all N0 and N1 columns of its 256 rows; the intermediate P never leaves the chip):
//
//   warp 0      TMA producer, in both CTAs: its own 128 rows of each A chunk, its own half
//               of the weights (once), completing on the LEADER CTA's barriers, which
//               count both CTAs' bytes
//   warp 1      TMEM (both CTAs allocate the pair's columns together); in the leader CTA
//               only, the MMA issuer for both: GEMM0 into TMEM, P (packed in place over
//               GEMM0's columns) -> GEMM1 in the TMEM-A form; its commits arrive on the
//               barriers of both CTAs at once
//   warps 2..9  epilogue, in both CTAs, two warpgroups taking alternate 256-row tiles:
//               D0 -> bias + act -> P in TMEM, then D1 -> bias + act -> the output rows
//               (coalesced stores, no staging tile); each warp reports to the leader's
//               barriers, so the leader's MMAs wait for both CTAs' epilogues
//
// Two 256-row tiles are in flight per pair: tile i uses TMEM buffer i & 1 (D0, then P and
// D1), and the MMA order is G0(0), G0(1), then G1(k), G1(k + 1), G0(k + 2), G0(k + 3).
// Limits (the host checks them): N0 and N1 multiples of 128 (each CTA's half a whole
// number of 64-wide blocks), two buffers of max(N0, N0 / 2 + N1) TMEM columns within 512,
// K0 at most kMaxW0Chunks * 64, row-major weights.
//
// Every wait is bounded; a CTA that gives up leaves its loops, and both CTAs meet at one
// cluster barrier before either exits, so neither releases shared memory or TMEM that the
// other may still read or signal.
#pragma once

#include "chain_kernel.cuh"

namespace b2b {
namespace B2B_KNS {

// Barrier slots (8 bytes each) at p.off_bar.  FULL, W0C, W1FULL, P_FULL, ACC_EMPTY,
// BIAS_READY and MMA_DONE are used in the leader CTA only (the peer's producer and
// epilogue arrive on the leader's copies); EMPTY, ACC_FULL and D1_FULL in both CTAs (the
// leader's MMA commits arrive on both copies at once).
enum : uint32_t {
  PB_FULL0 = 0,
  PB_EMPTY0 = kMaxStages,
  PB_W0C0 = 2 * kMaxStages,
  PB_W1FULL = PB_W0C0 + kMaxW0Chunks,
  PB_ACC_FULL0 = PB_W1FULL + 1,
  PB_D1_FULL0 = PB_ACC_FULL0 + 2,
  PB_P_FULL0 = PB_D1_FULL0 + 2,
  PB_ACC_EMPTY0 = PB_P_FULL0 + 2,
  PB_BIAS_READY = PB_ACC_EMPTY0 + 2,
  PB_MMA_DONE = PB_BIAS_READY + 1,
  PB_COUNT = PB_MMA_DONE + 1,
};
static_assert(8u * PB_COUNT + 8u <= kBarRegionBytes, "barrier region too small");

constexpr uint16_t kBothCtas = 3;   // CTA mask of a pair's commits

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// 256-row tiles of this pair: q, q + npairs, ...  (p.num_tiles counts 256-row tiles.)
__device__ __forceinline__ int cta2_tiles(const ChainParams& p) {
  const int q = static_cast<int>(cluster_id_x()), n = static_cast<int>(cluster_count_x());
  return q < p.num_tiles ? (p.num_tiles - 1 - q) / n + 1 : 0;
}
// First row of this CTA's 128 rows of the pair's it-th tile.
__device__ __forceinline__ int32_t cta2_row0(int it, uint32_t rank) {
  const int t = static_cast<int>(cluster_id_x() + static_cast<uint32_t>(it) * cluster_count_x());
  return t * 2 * kBlockM + static_cast<int32_t>(rank) * kBlockM;
}

__device__ __forceinline__ bool warp_wait_cl(bool alive, uint32_t bar, uint32_t parity,
                                             const ChainParams& p, volatile uint32_t* abort_flag,
                                             uint32_t site, int32_t t) {
  const bool ok = alive && mbar_wait_cluster(bar, parity, p.wait_limit_ns, abort_flag, p.err,
                                             p.kernel_id, site, t);
  return __all_sync(0xffffffffu, ok);
}

// Wait of the MMA issuer on a barrier that only TMA transactions complete (ring FULL,
// resident weights): both CTAs' loads of the pair signal the leader's barrier with their
// byte counts, and the MMAs that read the data go through the async proxy, so a CTA-scope
// acquire suffices (measured 1.5 % faster on the FFN-like chain than a cluster-scope one).
__device__ __forceinline__ bool warp_wait_tx(uint32_t bar, uint32_t parity, const ChainParams& p,
                                             volatile uint32_t* abort_flag, uint32_t site,
                                             int32_t t) {
  const bool ok = mbar_wait(bar, parity, p.wait_limit_ns, abort_flag, p.err, p.kernel_id, site, t);
  return __all_sync(0xffffffffu, ok);
}

// L2 prefetch of this CTA's 128 rows of the pair's it-th tile (warming only).
__device__ __forceinline__ void cta2_prefetch_rows(const ChainParams& p, int it, uint32_t rank) {
  const int32_t m0 = cta2_row0(it, rank);
  if (p.pf_a == nullptr || m0 >= p.M) return;
  const uint64_t off = static_cast<uint64_t>(m0) * p.pf_a_tile_bytes / kBlockM;
  const uint64_t n = min(static_cast<uint64_t>(p.pf_a_tile_bytes), p.pf_a_bytes - off);
  bulk_prefetch_l2(p.pf_a + off, static_cast<uint32_t>(n));
}

// ------------------------------------------------------------------------------------
// producer (both CTAs)
// ------------------------------------------------------------------------------------
__device__ void cta2_producer(const ChainParams& p, const CUtensorMap* tmA, const CUtensorMap* tmW0,
                              const CUtensorMap* tmW1, uint32_t base, uint32_t bars, uint32_t rank,
                              volatile uint32_t* abort_flag) {
  const uint32_t lead = elect_one();
  const bool leader = rank == 0;
  const uint64_t pol_stream = l2_policy_evict_first();
  const uint64_t pol_keep = l2_policy_evict_last();
  const int nb0 = p.N0p / 128, nb1 = p.N1p / 128;   // 64-wide blocks in each CTA's half
  auto leader_bar = [&](uint32_t slot) { return mapa_shared(bars + 8u * slot, 0u); };
  Tracer trace(p, 0, lead);
  grid_dependency_wait();   // global memory only after the previous grid has completed
  trace(EV_PROD_START, 0, 0);
  const int ntiles = cta2_tiles(p);
  int stage = 0;
  uint32_t phase = 0;
  uint32_t issued = 0, issued_parity = 0;   // leader: per stage, a fill in flight and its parity
  uint32_t w_issued = 0;                    // leader: W0 chunk barriers (bits 0..7), W1 (bit 8)
  bool ok = true;
  for (int it = 0; ok && it < ntiles; ++it) {
    const int32_t m0 = cta2_row0(it, rank);
    for (int kc = 0; kc < p.kchunks0; ++kc) {
      if (it == 0) {
        // this CTA's half of W0's chunk kc (once), beside the first tile's A chunk kc
        if (leader)
          mbar_arrive_expect_tx_if(lead, bars + 8u * (PB_W0C0 + kc), 2u * p.w0_chunk_bytes);
        tma_load_3d_pair(lead, base + p.off_w0 + kc * p.w0_chunk_bytes, tmW0,
                         leader_bar(PB_W0C0 + kc), 0, kc * kChunkK, static_cast<int32_t>(rank) * nb0,
                         pol_keep);
        w_issued |= 1u << kc;
      }
      if (!warp_mbar_wait(bars + 8u * (PB_EMPTY0 + stage), phase ^ 1u, p, abort_flag,
                          SITE_PRODUCER_EMPTY, m0)) {
        ok = false;
        break;
      }
      trace(EV_PROD_ACQUIRE, kc, it);
      if (leader)
        mbar_arrive_expect_tx_if(lead, bars + 8u * (PB_FULL0 + stage), 2u * kABytes);
      tma_load_2d_pair(lead, base + p.off_ring + stage * p.stage_bytes, tmA,
                       leader_bar(PB_FULL0 + stage), kc * kChunkK, m0, pol_stream);
      trace(EV_PROD_ISSUED, kc, it);
      issued |= 1u << stage;
      issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == static_cast<int>(p.num_stages)) { stage = 0; phase ^= 1u; }
    }
    if (ok && it == 0) {
      // this CTA's half of W1 (once), needed from the first GEMM1 on
      if (leader)
        mbar_arrive_expect_tx_if(lead, bars + 8u * PB_W1FULL,
                                 2u * static_cast<uint32_t>(p.kchunks1) * p.w1_chunk_bytes);
      for (int kc1 = 0; kc1 < p.kchunks1; ++kc1)
        tma_load_3d_pair(lead, base + p.off_w1 + kc1 * p.w1_chunk_bytes, tmW1,
                         leader_bar(PB_W1FULL), 0, kc1 * kChunkK,
                         static_cast<int32_t>(rank) * nb1, pol_keep);
      w_issued |= 1u << 8;
      trace(EV_PROD_W1_ISSUED, 0, it);
    }
  }
  if (!ok && leader) {
    // Gave up: let the fills in flight land (both CTAs' copies complete on these barriers)
    // before the pair can exit.
    const uint64_t drain_ns = 100000000ull;
    for (uint32_t s = 0; s < p.num_stages; ++s)
      if (issued & (1u << s))
        (void)mbar_wait_cluster(bars + 8u * (PB_FULL0 + s), (issued_parity >> s) & 1u, drain_ns,
                                nullptr, p.err, p.kernel_id, SITE_PRODUCER_DRAIN, 0);
    for (uint32_t c = 0; c < static_cast<uint32_t>(kMaxW0Chunks); ++c)
      if (w_issued & (1u << c))
        (void)mbar_wait_cluster(bars + 8u * (PB_W0C0 + c), 0u, drain_ns, nullptr, p.err,
                                p.kernel_id, SITE_PRODUCER_DRAIN, 0);
    if (w_issued & (1u << 8))
      (void)mbar_wait_cluster(bars + 8u * PB_W1FULL, 0u, drain_ns, nullptr, p.err, p.kernel_id,
                              SITE_PRODUCER_DRAIN, 0);
  }
}

// ------------------------------------------------------------------------------------
// MMA issuer (leader CTA, one warp; the elected lane issues for the pair)
// ------------------------------------------------------------------------------------
template <bool BF16>
__device__ void cta2_mma(const ChainParams& p, uint32_t base, uint32_t bars, uint32_t tmem_base,
                         volatile uint32_t* abort_flag) {
  const uint32_t lead = elect_one();
  const uint32_t dt = BF16 ? 1u : 0u;
  // M = 256 over the pair; B (the weights, row-major) is MN-major.
  const uint32_t idesc0 = idesc_f16_f32(dt, 1u, 2 * kBlockM, p.N0p);
  const uint32_t idesc1 = idesc_f16_f32(dt, 1u, 2 * kBlockM, p.N1p);
  const uint64_t ring_a = sdesc_sw128(base + p.off_ring, 16u, 1024u);
  const uint64_t res_w0 = sdesc_sw128(base + p.off_w0, 8192u, 1024u);
  const uint64_t res_w1 = sdesc_sw128(base + p.off_w1, 8192u, 1024u);
  const uint32_t nb0 = static_cast<uint32_t>(p.N0p / 128);
  const uint64_t ones_desc = sdesc_sw128(base + p.off_bias, 16u, 0u);
  const uint64_t bias0_desc = sdesc_sw128(base + p.off_bias + kOnesBytes, kBiasBlockBytes, 1024u);
  const uint64_t bias1_desc =
      sdesc_sw128(base + p.off_bias + kOnesBytes + nb0 * kBiasBlockBytes, kBiasBlockBytes, 1024u);
  const uint32_t stage_step = p.stage_bytes >> 4;
  const uint32_t w0_step = p.w0_chunk_bytes >> 4, w1_step = p.w1_chunk_bytes >> 4;
  constexpr uint64_t kAStep = 32u >> 4, kBStep = 2048u >> 4;   // per 16-wide K step
  const int last_rem = p.K0 - (p.kchunks0 - 1) * kChunkK;
  const int last_nks = last_rem >= 64 ? 4 : (last_rem + 15) >> 4;
  const int ntiles = cta2_tiles(p);
  Tracer trace(p, 1, lead, 3);
  bool ok = true, bias_ready = false, w1_ready = false;
  int stage = 0;
  uint32_t phase = 0;
  trace(EV_MMA_SETUP, 0, 0);
  grid_dependency_wait();
  trace(EV_DEP_READY, 0, 0);

  auto issue_g0 = [&](int it) -> bool {
    const uint32_t b = static_cast<uint32_t>(it) & 1u, use = (static_cast<uint32_t>(it) >> 1) & 1u;
    // both CTAs' epilogues have drained the buffer's previous tile (its D1)
    if (!warp_wait_cl(true, bars + 8u * (PB_ACC_EMPTY0 + b), use ^ 1u, p, abort_flag,
                      SITE_MMA_ACC_EMPTY, it))
      return false;
    trace(EV_MMA_ACC_FREE, b, it);
    tc_fence_after_sync();
    const uint32_t d0 = tmem_base + p.d0_col[b];
    for (int kc = 0; kc < p.kchunks0; ++kc) {
      if (it == 0 && !warp_wait_tx(bars + 8u * (PB_W0C0 + kc), 0u, p, abort_flag,
                                   SITE_MMA_WEIGHTS, it))
        return false;
      trace(EV_MMA_WAIT, kc, it);
      if (!warp_wait_tx(bars + 8u * (PB_FULL0 + stage), phase, p, abort_flag, SITE_MMA_FULL, it))
        return false;
      trace(EV_MMA_FULL, kc, it);
      const uint64_t adesc = ring_a + static_cast<uint64_t>(stage) * stage_step;
      const uint64_t bdesc = res_w0 + static_cast<uint64_t>(kc) * w0_step;
      const int nks = kc == p.kchunks0 - 1 ? last_nks : 4;
      for (int ks = 0; ks < nks; ++ks)
        mma_pair_ss(lead, d0, adesc + ks * kAStep, bdesc + ks * kBStep, idesc0,
                    (kc == 0 && ks == 0) ? 0u : 1u);
      trace(EV_MMA_ISSUED, kc, it);
      mma_commit_pair(lead, bars + 8u * (PB_EMPTY0 + stage), kBothCtas);   // frees both slots
      if (++stage == static_cast<int>(p.num_stages)) { stage = 0; phase ^= 1u; }
    }
    if (!bias_ready) {
      if (!warp_wait_cl(true, bars + 8u * PB_BIAS_READY, 0u, p, abort_flag, SITE_MMA_WEIGHTS, it))
        return false;
      bias_ready = true;
    }
    mma_pair_ss(lead, d0, ones_desc, bias0_desc, idesc0, 1u);   // D0 += bias
    mma_commit_pair(lead, bars + 8u * (PB_ACC_FULL0 + b), kBothCtas);
    trace(EV_MMA_G0_DONE, b, it);
    return true;
  };

  auto issue_g1 = [&](int j) -> bool {
    const uint32_t b = static_cast<uint32_t>(j) & 1u, use = (static_cast<uint32_t>(j) >> 1) & 1u;
    // both CTAs' P (packed into their TMEM) is complete
    if (!warp_wait_cl(true, bars + 8u * (PB_P_FULL0 + b), use, p, abort_flag, SITE_MMA_P_FULL, j))
      return false;
    trace(EV_MMA_P_READY, b, j);
    tc_fence_after_sync();
    if (!w1_ready) {
      if (!warp_wait_tx(bars + 8u * PB_W1FULL, 0u, p, abort_flag, SITE_MMA_WEIGHTS, j))
        return false;
      w1_ready = true;
      trace(EV_MMA_W1_FULL, 0, j);
    }
    const uint32_t d1 = tmem_base + p.d1_col[b];
    const uint32_t a0 = tmem_base + p.d0_col[b];   // P: 8 packed columns per 16-wide K step
    const int rem1 = p.N0p - (p.kchunks1 - 1) * kChunkK;
    const int last_nks1 = rem1 >= 64 ? 4 : (rem1 >> 4);
    for (int kc1 = 0; kc1 < p.kchunks1; ++kc1) {
      const uint64_t bdesc = res_w1 + static_cast<uint64_t>(kc1) * w1_step;
      const int nks = kc1 == p.kchunks1 - 1 ? last_nks1 : 4;
      for (int ks = 0; ks < nks; ++ks)
        mma_pair_ts(lead, d1, a0 + 32u * static_cast<uint32_t>(kc1) + 8u * static_cast<uint32_t>(ks),
                    bdesc + ks * kBStep, idesc1, (kc1 == 0 && ks == 0) ? 0u : 1u);
      trace(EV_MMA_ISSUED, 8 + kc1, j);
    }
    mma_pair_ss(lead, d1, ones_desc, bias1_desc, idesc1, 1u);   // D1 += bias
    mma_commit_pair(lead, bars + 8u * (PB_D1_FULL0 + b), kBothCtas);
    trace(EV_MMA_G1_DONE, b, j);
    return true;
  };

  for (int it = 0; ok && it < 2 && it < ntiles; ++it) ok = issue_g0(it);
  for (int k = 0; ok && k < ntiles; k += 2) {
    ok = issue_g1(k);
    if (ok && k + 1 < ntiles) ok = issue_g1(k + 1);
    if (ok && k + 2 < ntiles) ok = issue_g0(k + 2);
    if (ok && k + 3 < ntiles) ok = issue_g0(k + 3);
  }
  // Whatever happened, no MMA may still be running (reading either CTA's shared memory or
  // writing either CTA's TMEM) when the pair leaves.
  mma_commit_pair(lead, bars + 8u * PB_MMA_DONE, 1u);
  (void)mbar_wait(bars + 8u * PB_MMA_DONE, 0u, p.wait_limit_ns, nullptr, p.err, p.kernel_id,
                  SITE_MMA_DRAIN, 0);
  __syncwarp();
}

// ------------------------------------------------------------------------------------
// bias operands: this CTA's half of each GEMM's columns
// ------------------------------------------------------------------------------------
// As fill_bias_operands (the ONES tile, then per GEMM one 2 KiB BIAS block per 64-wide N
// block with the biases in k-row 0), over the columns [rank * N / 2, (rank + 1) * N / 2)
// that this CTA supplies to the pair's B operand.
__device__ __forceinline__ void fill_bias_half(const ChainParams& p, uint8_t* region, int tid,
                                               int nthreads, uint32_t rank) {
  const int nb0 = p.N0p / 128, nb1 = p.N1p / 128;
  const int c0 = static_cast<int>(rank) * (p.N0p / 2), c1 = static_cast<int>(rank) * (p.N1p / 2);
  uint32_t* words = reinterpret_cast<uint32_t*>(region);
  const int nwords = (static_cast<int>(kOnesBytes) + (nb0 + nb1) * static_cast<int>(kBiasBlockBytes)) >> 2;
  const uint32_t one = p.is_bf16 ? 0x3F80u : 0x3C00u;
  for (int w = tid; w < nwords; w += nthreads) {
    const int o = w << 2;
    if (o < static_cast<int>(kOnesBytes))
      words[w] = o == (o >> 7) * 144 ? one : 0u;   // row r: byte r * 128 + r * 16
    else if (((o - static_cast<int>(kOnesBytes)) & static_cast<int>(kBiasBlockBytes - 1)) >= 128)
      words[w] = 0u;
  }
  uint16_t* halves = reinterpret_cast<uint16_t*>(region + kOnesBytes);
  constexpr int kBlockHalves = static_cast<int>(kBiasBlockBytes / 2);
  for (int n = tid; n < nb0 * 64; n += nthreads) {
    const int col = c0 + n;
    halves[(n >> 6) * kBlockHalves + (n & 63)] =
        (col < p.N0 && p.b0 != nullptr) ? p.b0[col] : uint16_t(0);
  }
  for (int n = tid; n < nb1 * 64; n += nthreads) {
    const int col = c1 + n;
    halves[(nb0 + (n >> 6)) * kBlockHalves + (n & 63)] =
        (col < p.N1 && p.b1 != nullptr) ? p.b1[col] : uint16_t(0);
  }
}

// ------------------------------------------------------------------------------------
// epilogue (both CTAs; warpgroup g takes the pair's tiles i with i & 1 == g)
// ------------------------------------------------------------------------------------
template <bool BF16>
__device__ void cta2_epilogue(const ChainParams& p, const CUtensorMap* tmOut, uint32_t base,
                              uint32_t bars, uint32_t tmem_base, uint32_t rank,
                              volatile uint32_t* abort_flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = (warp - 2) >> 2;   // warpgroup = the tiles it takes
  const int q = warp & 3;          // TMEM lane quadrant this warp may access
  const uint32_t tm_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
  const bool elected = threadIdx.x == 64 + g * 128;
  auto leader_bar = [&](uint32_t slot) { return mapa_shared(bars + 8u * slot, 0u); };
  // Reports to the leader's barrier `slot` that this warp's TMEM accesses of the tile are
  // complete (its tcgen05.wait::ld / wait::st have returned and are fenced), releasing at
  // CTA scope: a release at cluster scope would first wait until this thread's global
  // stores of the output are performed cluster-wide, which the MMA issuer does not need
  // and which cost ~0.6 us per arrive.
  auto report = [&](uint32_t slot) { mbar_arrive_remote(leader_bar(slot)); };
  Tracer trace(p, 2u + static_cast<uint32_t>(g), elected ? 1u : 0u);
  // this warp's output staging slot (p.out_stage)
  const uint32_t slot = base + p.off_out[0] + static_cast<uint32_t>(warp - 2) * 4096u;
  bool alive = true;
  const int ntiles = cta2_tiles(p);
  for (int it = g; it < ntiles; it += 2) {
    const uint32_t b = static_cast<uint32_t>(it) & 1u, use = (static_cast<uint32_t>(it) >> 1) & 1u;
    const int32_t m0 = cta2_row0(it, rank);
    // GEMM0's accumulator -> bias (in it) + act -> P packed in place in TMEM
    alive = warp_wait_cl(alive, bars + 8u * (PB_ACC_FULL0 + b), use, p, abort_flag,
                         SITE_EPI_ACC_FULL, it);
    if (elected) trace(EV_EPI_ACC_READY, g, it);
    tc_fence_after_sync();
    if (alive) drain64_to_tmem<BF16>(p.act0, tm_lane, p.d0_col[b], p.N0p, p.d0_col[b]);
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) report(PB_P_FULL0 + b);
    if (elected) trace(EV_EPI_P_DONE, g, it);
    // GEMM1's accumulator -> act -> the output rows, coalesced (no staging tile: the ring
    // keeps that shared memory)
    alive = warp_wait_cl(alive, bars + 8u * (PB_D1_FULL0 + b), use, p, abort_flag,
                         SITE_EPI_D1_FULL, it);
    if (elected) trace(EV_EPI_D1_READY, g, it);
    tc_fence_after_sync();
    // The buffer (D0 -> P + D1) may take tile it + 2 as soon as the last TMEM load of the
    // tile has completed: the drain reports to the leader's ACC_EMPTY then, before it
    // converts and stores those columns from registers.
    if (alive && p.out_stage) {   // warp-uniform: TMEM loads and the slot are the warp's
      drain64_release_to_staging<BF16>(p.act1, tm_lane, p.d1_col[b], p.N1p, slot, tmOut,
                                       m0 + q * 32, p.M, lane, leader_bar(PB_ACC_EMPTY0 + b));
    } else if (alive) {   // warp-uniform: the drain's TMEM loads and shuffles are warp-collective
      drain64_release_to_global<BF16>(p.act1, tm_lane, p.d1_col[b], p.N1p, p.out_ptr,
                                      m0 + q * 32, p.M, p.out_ld, p.N1, lane,
                                      leader_bar(PB_ACC_EMPTY0 + b));
    } else {
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) report(PB_ACC_EMPTY0 + b);
    }
    if (elected) trace(EV_EPI_DRAINED, g, it);
    if (elected) trace(EV_EPI_STORED, g, it);
  }
  // the TMA engine has read every staged box before the CTA can leave
  if (p.out_stage && lane == 0) bulk_wait_read_all();
}

// ------------------------------------------------------------------------------------
// the kernel (launched in clusters of two CTAs)
// ------------------------------------------------------------------------------------
template <bool BF16>
__global__ void __launch_bounds__(kNumThreads, 1)
    chain_cta2_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmW0,
                      const __grid_constant__ CUtensorMap tmW1,
                      const __grid_constant__ CUtensorMap tmOut, const ChainParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t bars = base + p.off_bar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + p.off_bar + 8u * PB_COUNT);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const uint32_t rank = cluster_ctarank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Tracer ktrace(p, 1, threadIdx.x == 32 ? 1u : 0u);
  ktrace(EV_KERNEL_ENTRY, 0, 0);
  constexpr uint32_t kParamLines = (sizeof(ChainParams) + 63u) / 64u;
  if (threadIdx.x >= 64u && threadIdx.x < 64u + kParamLines) {
    const uint32_t w = reinterpret_cast<const uint32_t*>(&p)[(threadIdx.x - 64u) * 16u];
    asm volatile("" ::"r"(w));
  }

  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < p.num_stages; ++s) {
      mbar_init(bars + 8u * (PB_FULL0 + s), 1);
      mbar_init(bars + 8u * (PB_EMPTY0 + s), 1);
    }
    for (uint32_t c = 0; c < static_cast<uint32_t>(kMaxW0Chunks); ++c)
      mbar_init(bars + 8u * (PB_W0C0 + c), 1);
    mbar_init(bars + 8u * PB_W1FULL, 1);
    for (uint32_t b = 0; b < 2; ++b) {
      mbar_init(bars + 8u * (PB_ACC_FULL0 + b), 1);
      mbar_init(bars + 8u * (PB_D1_FULL0 + b), 1);
      mbar_init(bars + 8u * (PB_P_FULL0 + b), 2 * 4);       // four warps of one group, per CTA
      mbar_init(bars + 8u * (PB_ACC_EMPTY0 + b), 2 * 4);
    }
    mbar_init(bars + 8u * PB_BIAS_READY, 2 * kNumEpiWarps);
    mbar_init(bars + 8u * PB_MMA_DONE, 1);
    *abort_flag = 0u;
    fence_barrier_init();
    fence_proxy_async_smem();
    grid_launch_dependents();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmW0);
    tma_prefetch_desc(&tmW1);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), p.tmem_cols);
    tmem_relinquish_pair();
  }
  // Both CTAs' barriers are initialised and the pair's TMEM is allocated before either
  // CTA signals the other.
  tc_fence_before_sync();
  cluster_sync();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  ktrace(EV_SETUP_DONE, 0, 0);

  if (warp == 0) {
    // This CTA's rows of the first two tiles into L2 while the previous kernel finishes
    // (a hint only; see chain_kernel.cuh).  No further prefetches: prefetching tile it + 2
    // behind tile it's first chunk made the FFN-like chain 4 % slower (42.6 against 40.8
    // us at M = 262144), its bulk prefetches queueing beside the ring's own loads.
    if (lane == 0) {
      cta2_prefetch_rows(p, 0, rank);
      cta2_prefetch_rows(p, 1, rank);
    }
    __syncwarp();
    cta2_producer(p, &tmA, &tmW0, &tmW1, base, bars, rank, abort_flag);
    __syncwarp();
  } else if (warp == 1) {
    if (rank == 0) cta2_mma<BF16>(p, base, bars, tmem_base, abort_flag);
    __syncwarp();
  } else {
    grid_dependency_wait();
    fill_bias_half(p, base_ptr + p.off_bias, static_cast<int>(threadIdx.x) - 64, kNumEpiThreads,
                   rank);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive_cluster(mapa_shared(bars + 8u * PB_BIAS_READY, 0u));
    cta2_epilogue<BF16>(p, &tmOut, base, bars, tmem_base, rank, abort_flag);
  }

  // Neither CTA leaves while the other may still read its shared memory (the leader's
  // MMAs read the peer's operands) or arrive on its barriers.
  tc_fence_before_sync();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, p.tmem_cols);
  }
}

}  // namespace B2B_KNS
}  // namespace b2b
