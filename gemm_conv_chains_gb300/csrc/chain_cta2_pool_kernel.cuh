// chain_cta2_pool_kernel.cuh -- conv (R x S, stride 1, halo boxes) + bias + ReLU + 2x2
// max-pool over CTA pairs (tcgen05 .cta_group::2).
//
// The Welder notes' Conv + ReLU + MaxPool tile graph ("Tile-graph Scheduling", Figure 5)
// with the conv as an implicit GEMM whose N (the output channels) is small: with N = 64 an
// M128 x N64 x K16 MMA is short (48-51 cycles on one SM), and the one issuing thread's
// pauses between ring stages leave the tensor core idle.  Over a CTA pair one
// tcgen05.mma of M = 256 rows takes the first CTA's 8 x 16 output tile from its shared
// memory and the second CTA's tile from the second's, and B (the filters) columns
// [0, N/2) from the first CTA and [N/2, N) from the second: one instruction does both SMs'
// work (measured 43 cycles for M256 x N64 x K16), and each SM holds half of the filters,
// which leaves room for a deeper ring.
//
//   warp 0      TMA producer, in both CTAs: its own tile's halo boxes (one per column tap
//               and channel block, all row taps at once) and its half of the filters
//               (once), completing on the LEADER CTA's barriers, which count both CTAs'
//               bytes
//   warp 1      TMEM (both CTAs allocate the pair's columns together); in the leader CTA
//               only, an MMA issuer for both; its commits arrive on the barriers of both
//               CTAs at once
//   warps 10,11 in the leader CTA, the second and third MMA issuers (p.two_issuers = 1,
//               2): issuer j takes the pair-tiles i with i mod issuers = j from its own
//               sub-ring of the ring, so that the others issue while one waits
//   warps 2..9  epilogue, in both CTAs, two warpgroups taking alternate pair-tiles: the
//               CTA's own 128 accumulator rows + the bias (fp32) -> ReLU, rounding -> 2x2
//               max in registers -> a 4 x 8 pooled tile staged in shared memory -> TMA
//               store; each warp reports to the leader's barrier
//
// Pair q takes the pair-tiles q, q + pairs, ...; pair-tile u is the 8 x 16 output tiles 2u
// (first CTA) and 2u + 1 (second).  An odd tile count leaves the last pair-tile's second
// tile empty: its boxes lie past the last image (TMA reads zeros) and nothing is stored.
// Two accumulator buffers per issuer (four, or six with three issuers): the i-th
// pair-tile of the pair uses buffer i mod buffers.  Limits (the host checks them):
// stride 1, R > 1 (halo boxes), N0p <= 128, and three issuers only where six buffers fit
// the 512 TMEM columns.
//
// Every wait is bounded; a CTA that gives up leaves its loops, and both CTAs meet at one
// cluster barrier before either exits.
#pragma once

#include "chain_cta2_kernel.cuh"

namespace b2b {
namespace B2B_KNS {

// Barrier slots at p.off_bar.  FULL, WFULL, ACC_EMPTY and MMA_DONE are used in the leader
// CTA only; EMPTY and ACC_FULL in both (the leader's commits arrive on both).
enum : uint32_t {
  QB_FULL0 = 0,
  QB_EMPTY0 = kPool2MaxStages,
  QB_WFULL = 2 * kPool2MaxStages,
  QB_ACC_FULL0 = QB_WFULL + 1,
  QB_ACC_EMPTY0 = QB_ACC_FULL0 + kPool2MaxBufs,
  QB_MMA_DONE = QB_ACC_EMPTY0 + kPool2MaxBufs,
  QB_COUNT = QB_MMA_DONE + 1,
};
static_assert(8u * QB_COUNT + 8u <= kBarRegionBytes, "barrier region too small");

// MMA issuers, accumulator buffers, and the TMEM column of buffer b (buffers are
// p.d0_col[1] columns apart).
__device__ __forceinline__ int pool2_issuers(const ChainParams& p) { return 1 + p.two_issuers; }
__device__ __forceinline__ int pool2_bufs(const ChainParams& p) {
  return p.two_issuers == 2 ? 6 : 4;
}
__device__ __forceinline__ uint32_t pool2_col(const ChainParams& p, uint32_t b) {
  return b * static_cast<uint32_t>(p.d0_col[1]);
}

// Pair-tiles of the whole launch, and the number this pair processes.
__device__ __forceinline__ int pool2_pairtiles(const ChainParams& p) {
  return (p.num_tiles + 1) >> 1;
}
__device__ __forceinline__ int pool2_local(const ChainParams& p) {
  const int q = static_cast<int>(cluster_id_x()), n = static_cast<int>(cluster_count_x());
  const int total = pool2_pairtiles(p);
  return q < total ? (total - 1 - q) / n + 1 : 0;
}
// The tile of this CTA in the pair's i-th pair-tile.
__device__ __forceinline__ int32_t pool2_tile(int i, uint32_t rank) {
  const int32_t u = static_cast<int32_t>(cluster_id_x() + static_cast<uint32_t>(i) * cluster_count_x());
  return 2 * u + static_cast<int32_t>(rank);
}

// The sub-ring of issuer j of n: the ring's stages split as evenly as they go, issuer j
// owning [start, end) and walking it in order (SubRing), so that every slot has one
// consumer, never more than one phase ahead of its producer.
__device__ __forceinline__ SubRing pool2_subring(const ChainParams& p, int j) {
  const int n = pool2_issuers(p), S = static_cast<int>(p.num_stages);
  const int per = S / n, extra = S % n;
  const int start = j * per + min(j, extra);
  return make_subring(start, start + per + (j < extra ? 1 : 0));
}

// The bias of every output channel as fp32 (zero past N0, and with no bias), 256 words
// at `region`, one word per thread: the epilogue adds it to the accumulators.
__device__ __forceinline__ void fill_pool_bias(const ChainParams& p, float* region, int tid,
                                               int nthreads) {
  for (int n = tid; n < 256; n += nthreads) {
    float v = 0.0f;
    if (n < p.N0 && p.b0 != nullptr) {
      const uint16_t h = p.b0[n];
      v = p.is_bf16 ? __uint_as_float(static_cast<uint32_t>(h) << 16)
                    : __half2float(__ushort_as_half(h));
    }
    region[n] = v;
  }
}

__device__ void pool2_producer(const ChainParams& p, const CUtensorMap* tmA, const CUtensorMap* tmW0,
                               uint32_t base, uint32_t bars, uint32_t rank,
                               volatile uint32_t* abort_flag) {
  const uint32_t lead = elect_one();
  const bool leader = rank == 0;
  const uint64_t pol_stream = l2_policy_evict_first();
  const uint64_t pol_keep = l2_policy_evict_last();
  auto leader_bar = [&](uint32_t slot) { return mapa_shared(bars + 8u * slot, 0u); };
  Tracer trace(p, 0, lead);
  grid_dependency_wait();   // global memory only after the previous grid has completed
  trace(EV_PROD_START, 0, 0);
  // this CTA's half of the filters, once: rows [rank * N0p / 2, (rank + 1) * N0p / 2) of
  // every (tap, channel block) chunk
  if (leader)
    mbar_arrive_expect_tx_if(lead, bars + 8u * QB_WFULL,
                             2u * static_cast<uint32_t>(p.kchunks0) * p.w0_chunk_bytes);
  {
    KPos k;
    for (int kc = 0; kc < p.kchunks0; ++kc, k.next(p))
      tma_load_3d_pair(lead, base + p.off_w0 + kc * p.w0_chunk_bytes, tmW0,
                       leader_bar(QB_WFULL), k.cb * kChunkK, k.t,
                       static_cast<int32_t>(rank) * (p.N0p / 2), pol_keep);
  }
  const int ntiles = pool2_local(p), nis = pool2_issuers(p);
  // the walkers of the sub-rings of the current pair-tile's issuer (r0) and of the next
  SubRing r0 = pool2_subring(p, 0), r1 = pool2_subring(p, min(1, nis - 1)),
          r2 = pool2_subring(p, min(2, nis - 1));
  uint32_t issued = 0, issued_parity = 0;   // leader: per stage, a fill in flight and its parity
  bool ok = true;
  for (int i = 0; ok && i < ntiles; ++i) {
    const int32_t t = pool2_tile(i, rank);
    const TileCoord tc = tile_coord<true>(p, t);   // past the last tile: an image past the end
    KPos k;
    for (int kc = 0; kc < p.kstages0; ++kc, k.next_halo(p)) {
      const int stage = r0.slot;
      const uint32_t phase = r0.phase;
      if (!warp_mbar_wait(bars + 8u * (QB_EMPTY0 + stage), phase ^ 1u, p, abort_flag,
                          SITE_PRODUCER_EMPTY, t)) {
        ok = false;
        break;
      }
      trace(EV_PROD_ACQUIRE, kc, i);
      if (leader)
        mbar_arrive_expect_tx_if(lead, bars + 8u * (QB_FULL0 + stage), 2u * p.a_stage_bytes);
      tma_load_4d_pair(lead, base + p.off_ring + stage * p.stage_bytes, tmA,
                       leader_bar(QB_FULL0 + stage), k.cb * kChunkK, tc.wo0 + k.s - p.pad,
                       tc.ho0 - p.pad, tc.n, pol_stream);
      trace(EV_PROD_ISSUED, kc, i);
      issued |= 1u << stage;
      issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
      advance_subring(r0);
    }
    // the next pair-tile belongs to the next issuer
    if (nis == 2) {
      const SubRing x = r0;
      r0 = r1;
      r1 = x;
    } else if (nis == 3) {
      const SubRing x = r0;
      r0 = r1;
      r1 = r2;
      r2 = x;
    }
  }
  if (leader) {
    // Let the fills in flight land (both CTAs' copies complete on these barriers) before
    // the pair can exit: always the filters, and the ring when this producer gave up.
    const uint64_t drain_ns = 100000000ull;
    if (!ok)
      for (uint32_t s = 0; s < p.num_stages; ++s)
        if (issued & (1u << s))
          (void)mbar_wait_cluster(bars + 8u * (QB_FULL0 + s), (issued_parity >> s) & 1u,
                                  drain_ns, nullptr, p.err, p.kernel_id, SITE_PRODUCER_DRAIN, 0);
    (void)mbar_wait_cluster(bars + 8u * QB_WFULL, 0u, drain_ns, nullptr, p.err, p.kernel_id,
                            SITE_PRODUCER_DRAIN, 0);
  }
}

// Issuer `issuer` (0: warp 1; 1, 2: warps 10, 11, with p.two_issuers) of the leader CTA:
// it takes the pair-tiles i with i mod issuers = issuer, each into buffer i mod buffers,
// from its own sub-ring of the ring; the epilogue warpgroup of i's parity drains them.
template <bool BF16>
__device__ void pool2_mma(const ChainParams& p, uint32_t base, uint32_t bars, uint32_t tmem_base,
                          volatile uint32_t* abort_flag, int issuer) {
  const uint32_t lead = elect_one();
  const uint32_t dt = BF16 ? 1u : 0u;
  // M = 256 over the pair; the filters (B) are K-major.
  const uint32_t idesc0 = idesc_f16_f32(dt, 0u, 2 * kBlockM, p.N0p);
  const uint64_t ring_a = sdesc_sw128(base + p.off_ring, 16u, 1024u);
  const uint64_t res_w0 = sdesc_sw128(base + p.off_w0, 16u, 1024u);
  const uint32_t stage_step = p.stage_bytes >> 4;
  const uint32_t w0_step = p.w0_chunk_bytes >> 4;
  constexpr uint64_t kStep = 32u >> 4;   // per 16-wide K step, K-major A and B
  const int last_rem = p.K0 - (p.kc_per_tap - 1) * kChunkK;
  const int last_nks = last_rem >= 64 ? 4 : (last_rem + 15) >> 4;
  const int ntiles = pool2_local(p);
  const int nis = pool2_issuers(p), nbufs = pool2_bufs(p);
  Tracer trace(p, 1, issuer == 0 ? lead : 0u, 3);
  bool ok = true;
  SubRing ring = pool2_subring(p, issuer);   // this issuer's stages
  uint32_t b = static_cast<uint32_t>(issuer), use = 0u;   // buffer i mod nbufs, its parity
  trace(EV_MMA_SETUP, 0, 0);
  grid_dependency_wait();
  trace(EV_DEP_READY, 0, 0);
  ok = warp_wait_tx(bars + 8u * QB_WFULL, 0u, p, abort_flag, SITE_MMA_WEIGHTS, 0);
  for (int i = issuer; ok && i < ntiles; i += nis) {
    // both CTAs' epilogues have drained the buffer's previous pair-tile
    if (!warp_wait_cl(true, bars + 8u * (QB_ACC_EMPTY0 + b), use ^ 1u, p, abort_flag,
                      SITE_MMA_ACC_EMPTY, i)) {
      ok = false;
      break;
    }
    trace(EV_MMA_ACC_FREE, b, i);
    tc_fence_after_sync();
    const uint32_t d0 = tmem_base + pool2_col(p, b);
    int cb = 0, s_tap = 0;
    for (int kc = 0; kc < p.kstages0; ++kc) {
      const int stage = ring.slot;
      const uint32_t phase = ring.phase;
      trace(EV_MMA_WAIT, kc, i);
      if (!warp_wait_tx(bars + 8u * (QB_FULL0 + stage), phase, p, abort_flag, SITE_MMA_FULL, i)) {
        ok = false;
        break;
      }
      trace(EV_MMA_FULL, kc, i);
      const uint64_t adesc = ring_a + static_cast<uint64_t>(stage) * stage_step;
      const int nks = cb == p.kc_per_tap - 1 ? last_nks : 4;
      // The stage holds rows ho0 - pad .. + 8 + R - 1 (16 pixels each) of both tiles: row
      // tap r starts 16 rows = 2 KiB further in.
      for (int r = 0; r < p.R; ++r) {
        const int wchunk = (r * p.S + s_tap) * p.kc_per_tap + cb;
        const uint64_t a = adesc + static_cast<uint64_t>(r) * (2048u >> 4);
        const uint64_t w = res_w0 + static_cast<uint64_t>(wchunk) * w0_step;
        if (nks == 4) {
          mma_pair_ss_x4(lead, d0, a, w, kStep, kStep, idesc0, (kc == 0 && r == 0) ? 0u : 1u);
        } else {
          for (int ks = 0; ks < nks; ++ks)
            mma_pair_ss(lead, d0, a + ks * kStep, w + ks * kStep, idesc0,
                        (kc == 0 && r == 0 && ks == 0) ? 0u : 1u);
        }
      }
      trace(EV_MMA_ISSUED, kc, i);
      mma_commit_pair(lead, bars + 8u * (QB_EMPTY0 + stage), kBothCtas);   // frees both slots
      advance_subring(ring);
      if (++cb == p.kc_per_tap) { cb = 0; ++s_tap; }
    }
    if (!ok) break;
    mma_commit_pair(lead, bars + 8u * (QB_ACC_FULL0 + b), kBothCtas);
    trace(EV_MMA_G0_DONE, b, i);
    b += static_cast<uint32_t>(nis);
    if (b >= static_cast<uint32_t>(nbufs)) {
      b -= static_cast<uint32_t>(nbufs);
      use ^= 1u;
    }
  }
  // Whatever happened, no MMA may still be running (reading either CTA's shared memory or
  // writing either CTA's TMEM) when the pair leaves.
  mma_commit_pair(lead, bars + 8u * QB_MMA_DONE, 1u);
  (void)mbar_wait(bars + 8u * QB_MMA_DONE, 0u, p.wait_limit_ns, nullptr, p.err, p.kernel_id,
                  SITE_MMA_DRAIN, 0);
  __syncwarp();
}

// The CTA's 128 accumulator rows (the conv sums) of one pair-tile + the bias -> ReLU,
// rounding -> 2x2 max -> the 4 x 8 pooled tile, 32 columns at a time (as drain_pool, with
// the bias, 256 fp32 words at `bias`, added in fp32 before the rounding).
template <bool BF16>
__device__ __noinline__ void drain_pool_bias(uint32_t tm_lane, uint32_t col0, int ncols,
                                             uint32_t bias, uint32_t tile, int q, int lane) {
  const bool owner = (lane & 17) == 0;
  const int prow = q * 8 + (lane >> 1);
  for (int c = 0; c < ncols; c += 32) {
    const bool two = c + 16 < ncols;
    uint32_t a[16], b[16], v[8], w[8];
    tmem_ld32(tm_lane + col0 + c, two, a, b);
    float fa[16], fb[16];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 x = ld_shared_f4(bias + 4u * static_cast<uint32_t>(c + 4 * j));
      const float4 y = ld_shared_f4(bias + 4u * static_cast<uint32_t>(c + 16 + 4 * j));
      fa[4 * j] = x.x, fa[4 * j + 1] = x.y, fa[4 * j + 2] = x.z, fa[4 * j + 3] = x.w;
      fb[4 * j] = y.x, fb[4 * j + 1] = y.y, fb[4 * j + 2] = y.z, fb[4 * j + 3] = y.w;
    }
    tmem_wait_ld(a, b);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[j] = pack2<BF16, true>(__uint_as_float(a[2 * j]) + fa[2 * j],
                               __uint_as_float(a[2 * j + 1]) + fa[2 * j + 1]);
      w[j] = pack2<BF16, true>(__uint_as_float(b[2 * j]) + fb[2 * j],
                               __uint_as_float(b[2 * j + 1]) + fb[2 * j + 1]);
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

template <bool BF16>
__device__ void pool2_epilogue(const ChainParams& p, const CUtensorMap* tmOut, uint32_t base,
                               uint32_t bars, uint32_t tmem_base, uint32_t rank,
                               volatile uint32_t* abort_flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = (warp - 2) >> 2;   // warpgroup = the pair-tiles it takes
  const int q = warp & 3;          // TMEM lane quadrant this warp may access
  const uint32_t tm_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
  const bool elected = threadIdx.x == 64 + g * 128;
  const uint32_t bar_id = 2u + static_cast<uint32_t>(g);   // named barrier of the group
  auto leader_bar = [&](uint32_t slot) { return mapa_shared(bars + 8u * slot, 0u); };
  Tracer trace(p, 2u + static_cast<uint32_t>(g), elected ? 1u : 0u);
  const uint32_t out_tile = base + p.off_out[g];
  const int nch = (p.N0p + 63) >> 6;
  bool alive = true;
  const int ntiles = pool2_local(p), nbufs = pool2_bufs(p);
  const uint32_t bias = base + p.off_bias;
  uint32_t b = static_cast<uint32_t>(g), use = 0u;   // buffer i mod nbufs, its parity
  for (int i = g; i < ntiles; i += 2) {
    const int32_t t = pool2_tile(i, rank);
    const TileCoord tc = tile_coord<true>(p, t);
    alive = warp_wait_cl(alive, bars + 8u * (QB_ACC_FULL0 + b), use, p, abort_flag,
                         SITE_EPI_ACC_FULL, t);
    if (elected) trace(EV_EPI_ACC_READY, g, i);
    tc_fence_after_sync();
    if (elected) bulk_wait_read_all();   // this group's staging is free again
    named_bar_sync(bar_id, 128u);
    if (elected) trace(EV_EPI_STAGING, g, i);
    if (alive) drain_pool_bias<BF16>(tm_lane, pool2_col(p, b), p.N0p, bias, out_tile, q, lane);
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive_remote(leader_bar(QB_ACC_EMPTY0 + b));
    fence_proxy_async_smem();
    named_bar_sync(bar_id, 128u);
    if (elected && alive && t < p.num_tiles && !*abort_flag) {
      for (int nc = 0; nc < nch; ++nc)
        tma_store_4d(tmOut, out_tile + nc * kPoolChunkBytes, nc * 64, tc.wo0 >> 1, tc.ho0 >> 1,
                     tc.n);
      bulk_commit_group();
      trace(EV_EPI_STORED, g, i);
    }
    b += 2u;
    if (b >= static_cast<uint32_t>(nbufs)) {
      b -= static_cast<uint32_t>(nbufs);
      use ^= 1u;
    }
  }
  // the TMA engine has read every staged tile before the CTA can leave
  if (elected) bulk_wait_read_all();
}

// Warps 10 and 11 are the leader's second and third MMA issuers (p.two_issuers).
constexpr int kPool2Threads = kNumThreads + 64;

template <bool BF16>
__global__ void __launch_bounds__(kPool2Threads, 1)
    chain_cta2_pool_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmW0,
                           const __grid_constant__ CUtensorMap tmW1,
                           const __grid_constant__ CUtensorMap tmOut, const ChainParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t bars = base + p.off_bar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + p.off_bar + 8u * QB_COUNT);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const uint32_t rank = cluster_ctarank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  (void)tmW1;
  Tracer ktrace(p, 1, threadIdx.x == 32 ? 1u : 0u);
  ktrace(EV_KERNEL_ENTRY, 0, 0);
  constexpr uint32_t kParamLines = (sizeof(ChainParams) + 63u) / 64u;
  if (threadIdx.x >= 64u && threadIdx.x < 64u + kParamLines) {
    const uint32_t w = reinterpret_cast<const uint32_t*>(&p)[(threadIdx.x - 64u) * 16u];
    asm volatile("" ::"r"(w));
  }

  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < p.num_stages; ++s) {
      mbar_init(bars + 8u * (QB_FULL0 + s), 1);
      mbar_init(bars + 8u * (QB_EMPTY0 + s), 1);
    }
    mbar_init(bars + 8u * QB_WFULL, 1);
    for (int b = 0; b < pool2_bufs(p); ++b) {
      mbar_init(bars + 8u * (QB_ACC_FULL0 + b), 1);
      mbar_init(bars + 8u * (QB_ACC_EMPTY0 + b), 2 * 4);   // four warps of one group, per CTA
    }
    mbar_init(bars + 8u * QB_MMA_DONE, static_cast<uint32_t>(pool2_issuers(p)));
    *abort_flag = 0u;
    fence_barrier_init();
    fence_proxy_async_smem();
    grid_launch_dependents();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmW0);
    tma_prefetch_desc(&tmOut);
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
    pool2_producer(p, &tmA, &tmW0, base, bars, rank, abort_flag);
    __syncwarp();
  } else if (warp == 1) {
    if (rank == 0) pool2_mma<BF16>(p, base, bars, tmem_base, abort_flag, 0);
    __syncwarp();
  } else if (warp >= kSecondIssuerWarp) {
    const int issuer = warp - kSecondIssuerWarp + 1;
    if (rank == 0 && issuer < pool2_issuers(p))
      pool2_mma<BF16>(p, base, bars, tmem_base, abort_flag, issuer);
    __syncwarp();
  } else {
    grid_dependency_wait();
    fill_pool_bias(p, reinterpret_cast<float*>(base_ptr + p.off_bias),
                   static_cast<int>(threadIdx.x) - 64, kNumEpiThreads);
    named_bar_sync(4u, kNumEpiThreads);   // the bias words are written before any is read
    pool2_epilogue<BF16>(p, &tmOut, base, bars, tmem_base, rank, abort_flag);
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
