// api.cu -- the extern "C" entry points of libb2b.so (declared in include/b2b.h).
//
// Host side only: argument validation (before anything touches the GPU), TMA tensor-map
// encoding (cached), the shared-memory plan of each launch, and the launch itself on the
// caller's stream.  No device memory is allocated here.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <initializer_list>
#include <map>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "b2b.h"
#include "ptx.cuh"
#include "launch.h"

// The tile-graph model's ranking of a problem's layouts (defined with the plan functions).
static b2b_status model_top(const std::vector<int64_t>& key, std::vector<int32_t>* top);

namespace b2b {
namespace {

// ------------------------------------------------------------------------------------
// device state
// ------------------------------------------------------------------------------------
__device__ uint32_t g_error_word[4];   // {code, kernel id, wait site, tile}

constexpr int kMaxDevices = 64;
constexpr uint32_t kSmemLimit = 227u * 1024u;          // dynamic smem per CTA on sm_100/103
constexpr uint64_t kDefaultWaitNs = 1000000000ull;     // 1 s

struct DeviceState {
  std::once_flag once;
  int num_sms = 0;
  uint32_t* err = nullptr;                    // device address of g_error_word
  cudaError_t init_error = cudaSuccess;
  // bit 2 (v + V_COUNT traced) + bf16 of the pair of words: smem attribute set
  std::atomic<uint64_t> attr_done[2] = {0, 0};
  // CTA-pair kernel: resident clusters of two (per bf16 + 2 * traced), for the dynamic
  // shared memory size they were computed for; 0 = not yet known
  // per pair kernel (+4: conv + pool), dtype (+1: bf16) and build (+2: traced)
  std::atomic<int> cta2_clusters[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  std::atomic<size_t> cta2_smem[8] = {0, 0, 0, 0, 0, 0, 0, 0};
};
DeviceState g_dev[kMaxDevices];
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};

// Optional event trace (b2b_set_trace): caller-owned device buffer, read by later launches.
std::mutex g_trace_mu;
unsigned long long* g_trace_buf = nullptr;
uint32_t g_trace_cap = 0, g_trace_cta = 0;

DeviceState* device_state(b2b_status* st) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    *st = B2B_ERR_CUDA;
    return nullptr;
  }
  DeviceState& d = g_dev[dev];
  std::call_once(d.once, [&d, dev] {
    int n = 0;
    d.init_error = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (d.init_error == cudaSuccess) {
      d.num_sms = n;
      // The device address of the error word, with this device current.
      d.init_error = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err), g_error_word);
    }
    if (d.init_error != cudaSuccess) cudaGetLastError();
  });
  if (d.init_error != cudaSuccess) {
    *st = B2B_ERR_CUDA;
    return nullptr;
  }
  return &d;
}

// ------------------------------------------------------------------------------------
// TMA tensor maps
// ------------------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

struct MapKey {
  const void* ptr;
  uint32_t rank, is_bf16;
  uint64_t dims[4];
  uint64_t strides[3];
  uint32_t box[4];
  uint32_t elem_strides[4];
  uint32_t swizzle128, pad;
  bool operator==(const MapKey& o) const { return std::memcmp(this, &o, sizeof(MapKey)) == 0; }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    const uint64_t* w = reinterpret_cast<const uint64_t*>(&k);
    uint64_t h = 1469598103934665603ull;
    for (size_t i = 0; i < sizeof(MapKey) / 8; ++i) h = (h ^ w[i]) * 1099511628211ull;
    return static_cast<size_t>(h);
  }
};
std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;

// A tiled, 128B-swizzled (or, with swizzle128 false, unswizzled: the box lands densely,
// dimension 0 fastest) map with zero fill outside the tensor.  dims[0] is the contiguous
// dimension; strides are in bytes for dims 1..rank-1.  elem_strides: the box takes every
// elem_strides[i]-th element along dimension i (box[i] / elem_strides[i] of them land in
// shared memory).
bool make_map(CUtensorMap* out, const void* ptr, int is_bf16, uint32_t rank,
              std::initializer_list<uint64_t> dims, std::initializer_list<uint64_t> strides,
              std::initializer_list<uint32_t> box,
              std::initializer_list<uint32_t> elem_strides = {1, 1, 1, 1},
              bool swizzle128 = true) {
  MapKey key;
  std::memset(&key, 0, sizeof(key));
  key.swizzle128 = swizzle128 ? 1u : 0u;
  key.ptr = ptr;
  key.rank = rank;
  key.is_bf16 = static_cast<uint32_t>(is_bf16);
  std::copy(dims.begin(), dims.end(), key.dims);
  std::copy(strides.begin(), strides.end(), key.strides);
  std::copy(box.begin(), box.end(), key.box);
  std::copy(elem_strides.begin(), elem_strides.end(), key.elem_strides);
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    auto it = g_maps.find(key);
    if (it != g_maps.end()) {
      *out = it->second;
      return true;
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t gdim[4], gstride[3];
  cuuint32_t bdim[4], estride[4] = {1, 1, 1, 1};
  for (uint32_t i = 0; i < rank; ++i) {
    gdim[i] = key.dims[i];
    bdim[i] = key.box[i];
    estride[i] = key.elem_strides[i] != 0 ? key.elem_strides[i] : 1u;
  }
  for (uint32_t i = 0; i + 1 < rank; ++i) gstride[i] = key.strides[i];
  CUtensorMap m;
  const CUresult r = fn(&m, is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        rank, const_cast<void*>(ptr), gdim, gstride, bdim, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> lk(g_map_mu);
  if (g_maps.size() > 4096) g_maps.clear();
  g_maps.emplace(key, m);
  *out = m;
  return true;
}

// ------------------------------------------------------------------------------------
// helpers
// ------------------------------------------------------------------------------------
inline uint32_t round_up(uint32_t x, uint32_t m) { return (x + m - 1) / m * m; }
inline int32_t ceil_div(int64_t a, int64_t b) { return static_cast<int32_t>((a + b - 1) / b); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned2(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 1u) == 0; }
inline uint32_t pow2_at_least(uint32_t x) {
  uint32_t p = 32;
  while (p < x) p <<= 1;
  return p;
}
inline bool valid_dtype(int dt) { return dt == B2B_F16 || dt == B2B_BF16; }
inline bool valid_epi(int e) {
  return e == B2B_EPI_NONE || e == B2B_EPI_RELU || e == B2B_EPI_HARDSWISH;
}

// Byte sizes of the shared-memory regions of one launch (for the plan and its checks).
struct Regions {
  uint32_t ring, w_res, p_each, out_each, bias, bar;
  int32_t cand = 0, ncand = 0;   // the layout taken, as an index into the feasible ones
  uint32_t extend = 0;           // ring stages that may run on into the output staging
};

// TMEM columns of the accumulators.  Chain: nbuf D0 buffers of round_up(N0p, 32) columns,
// then nbuf D1 buffers of round_up(N1p, 32) columns (every buffer starts on a multiple of
// 32 columns); single/pool: two accumulator buffers, or four when nbuf is 4.  Returns the
// power-of-two allocation.
uint32_t tmem_layout(ChainParams& p, int mode, uint32_t nbuf, bool p_tmem = false) {
  const uint32_t s0 = round_up(static_cast<uint32_t>(p.N0p), 32u);
  for (uint32_t b = 0; b < kMaxBufs; ++b) p.d0_col[b] = p.d1_col[b] = 0;
  p.d2_col[0] = p.d2_col[1] = 0;
  p.pt_col[0] = p.pt_col[1] = 0;
  p.p_split = 0;
  p.p_hi = 0;
  if (mode == MODE_CHAIN && p_tmem && p.N0p > 256) {
    // Wide: all 512 columns.  GEMM0 runs over the halves of N0 into [0, 256) and
    // [256, 256 + N0p - 256); each half's P packs in place into its first 128 columns.  D1
    // sits in the upper columns of the half computed first: [128, 128 + N1p) on even tiles
    // (lower half first), [384, 384 + N1p) on odd ones (upper half first), so that a
    // tile's first GEMM0 pass never touches the previous tile's D1.
    p.p_split = 256u;
    p.p_hi = 256u;
    p.d0_col[0] = p.pt_col[0] = 0;
    p.d0_col[1] = p.pt_col[1] = 256u;
    p.d1_col[0] = 128u;
    p.d1_col[1] = 384u;
    return 512u;
  }
  if (mode == MODE_CHAIN3) {
    // Two buffers of D0, D1, D2 each: tile i uses buffer i & 1.
    const uint32_t s1 = round_up(static_cast<uint32_t>(p.N1p), 32u);
    const uint32_t s2 = round_up(static_cast<uint32_t>(p.N2p), 32u);
    for (uint32_t b = 0; b < 2; ++b) {
      p.d0_col[b] = b * s0;
      p.d1_col[b] = 2u * s0 + b * s1;
      p.d2_col[b] = 2u * (s0 + s1) + b * s2;
    }
    return pow2_at_least(2u * (s0 + s1 + s2));
  }
  if (mode == MODE_CHAIN && p_tmem && p.two_issuers) {
    // Two issuers: D0, P and D1 of both buffers apart -- [D0 0][D0 1][P 0][P 1][D1 0][D1 1]
    // -- so that an issuer's next GEMM0 overwrites nothing its GEMM1 or the epilogue may
    // still read.
    const uint32_t sp = round_up(static_cast<uint32_t>(p.N0p) / 2u, 32u);
    const uint32_t s1 = round_up(static_cast<uint32_t>(p.N1p), 32u);
    for (uint32_t b = 0; b < 2; ++b) {
      p.d0_col[b] = b * s0;
      p.pt_col[b] = 2u * s0 + b * sp;
      p.d1_col[b] = 2u * (s0 + sp) + b * s1;
    }
    return pow2_at_least(2u * (s0 + sp + s1));
  }
  if (mode == MODE_CHAIN && p_tmem) {
    // Buffer b holds D0, then P (packed, N0p / 2 columns, over D0) and D1 after it.
    const uint32_t d1off = round_up(static_cast<uint32_t>(p.N0p) / 2u, 32u);
    const uint32_t buf = round_up(std::max(s0, d1off + static_cast<uint32_t>(p.N1p)), 32u);
    p.d0_col[0] = p.pt_col[0] = 0;
    p.d0_col[1] = p.pt_col[1] = buf;
    p.d1_col[0] = d1off;
    p.d1_col[1] = buf + d1off;
    return pow2_at_least(2u * buf);
  }
  if (mode == MODE_CHAIN) {
    const uint32_t s1 = round_up(static_cast<uint32_t>(p.N1p), 32u);
    for (uint32_t b = 0; b < nbuf; ++b) {
      p.d0_col[b] = b * s0;
      p.d1_col[b] = nbuf * s0 + b * s1;
    }
    return pow2_at_least(nbuf * (s0 + s1));
  }
  // single / pool: nbuf (2 or 4) accumulator buffers
  const uint32_t n = nbuf >= 4u ? 4u : 2u;
  const uint32_t cols = pow2_at_least(n * s0);
  for (uint32_t b = 0; b < n; ++b) p.d0_col[b] = b * (cols / n);
  return cols;
}

// Shared-memory plan: ring of A (and, when streamed, weight) chunks; resident weights;
// P tiles; output staging; bias operands; barriers.  The candidates that leave at least two
// ring stages are feasible, in order of preference -- more tiles in flight, resident
// weights, separate staging.  `forced` >= 0 takes that feasible candidate (launches always
// name one: the tile-graph model's pick, a pinned or a measured choice); without it the
// first feasible one with three or more stages is taken (else the first feasible one),
// which only validation uses.  Fills p's layout fields.
bool plan_smem(ChainParams& p, int mode, bool w0mn, bool w1mn, size_t* smem_bytes,
               Regions* regions, int forced = -1) {
  const uint32_t budget = kSmemLimit - 1024u;   // 1 KiB slack to align the base to 1024
  const uint32_t n0blk = static_cast<uint32_t>((p.N0p + 63) / 64);
  const uint32_t n1blk = static_cast<uint32_t>((p.N1p + 63) / 64);
  // (Wide chains stream W0 by halves of N0: four 64-wide blocks per chunk.)
  const bool wide = mode == MODE_CHAIN && p.N0p > 256;
  p.w0_chunk_bytes = w0mn ? std::min(n0blk, wide ? 4u : n0blk) * 8192u
                          : static_cast<uint32_t>(p.N0p) * 128u;
  p.w1_chunk_bytes = mode == MODE_CHAIN ? (w1mn ? n1blk * 8192u : static_cast<uint32_t>(p.N1p) * 128u) : 0u;
  const uint32_t p_bytes = mode == MODE_CHAIN ? n0blk * kPChunkBytes : 0u;
  const uint32_t out_bytes = mode == MODE_CHAIN    ? n1blk * kPChunkBytes
                             : mode == MODE_SINGLE ? n0blk * kPChunkBytes
                                                   : n0blk * kPoolChunkBytes;
  // (the two-issuer conv chain: one slot of 32 rows x 16 columns per epilogue warp)
  const uint32_t slot_bytes = static_cast<uint32_t>(kNumEpiWarps) * kOutSlotBytes;
  // Bias operands: the ONES tile, then one BIAS block per 64-wide N block of each GEMM.
  const uint32_t bias_bytes =
      kOnesBytes + kBiasBlockBytes * (n0blk + (mode == MODE_CHAIN ? n1blk : 0u));
  const uint32_t bar_bytes = 1024u;
  const uint32_t w_res = static_cast<uint32_t>(p.kchunks0) * p.w0_chunk_bytes +
                         static_cast<uint32_t>(p.kchunks1) * p.w1_chunk_bytes;

  // Candidates in order of preference.  Chains: two tiles in flight with P in shared
  // memory; else two tiles in flight with P in TMEM (wide N0, where two P tiles and two
  // accumulator pairs do not fit); else one tile at a time.
  // dual: chain accumulator / P buffers (1, 2 or 4); single/pool always have two.
  // w0res: P in TMEM with W0 alone resident (row-major weights, at most kMaxW0Chunks K
  // chunks): the ring carries A and W1 chunks and the output goes from registers straight
  // to global memory, so the plan has no output staging.
  // two: (convs with halo boxes, N0 <= 64) two MMA issuers over two sub-rings that each
  // hold a whole tile's stages, resident filters, P in TMEM apart from D0 and D1, and the
  // output staged 16 columns at a time in a 1 KiB slot per epilogue warp, so that the ring
  // has room for both sub-rings.
  struct Cand { int dual, groups, resident, alias, p_tmem, w0res = 0, two = 0; };
  Cand cands[16];
  int ncand = 0;
  if (mode == MODE_CHAIN) {
    ChainParams probe = p;
    probe.two_issuers = 0;
    const bool tmem_quad_ok = tmem_layout(probe, mode, 4u) <= 512u;
    const bool tmem_dual_ok = tmem_layout(probe, mode, 2u) <= 512u;
    const bool tmem_p_ok = tmem_layout(probe, mode, 2u, true) <= 512u;
    probe.two_issuers = 1;
    const bool tmem_two_ok = tmem_layout(probe, mode, 2u, true) <= 512u;
    if (p.N0p > 256) {
      // Wide (256 < N0 <= 512, N1 <= 128): one tile in flight, P in TMEM, both
      // warpgroups on every tile, weights streamed.
      if (p.N1p <= 128) cands[ncand++] = {1, 1, 0, 0, 1};
    } else {
      if (p.R > 1 && p.stride == 1 && p.N0p <= 64 && tmem_two_ok)
        cands[ncand++] = {2, 2, 1, 0, 1, 0, 1};
      // Four tiles in flight (narrow chains): each epilogue group one tile ahead.
      if (tmem_quad_ok)
        for (int resident = 1; resident >= 0; --resident) cands[ncand++] = {4, 2, resident, 0, 0};
      if (tmem_dual_ok)
        for (int resident = 1; resident >= 0; --resident)
          for (int alias = 0; alias <= 1; ++alias) cands[ncand++] = {2, 2, resident, alias, 0};
      if (tmem_p_ok) {
        cands[ncand++] = {2, 2, 1, 0, 1};
        cands[ncand++] = {2, 2, 0, 0, 1};
        if (w0mn && w1mn && p.kchunks0 <= kMaxW0Chunks) cands[ncand++] = {2, 2, 0, 0, 1, 1};
      }
      for (int resident = 1; resident >= 0; --resident)
        for (int alias = 0; alias <= 1; ++alias) cands[ncand++] = {1, 1, resident, alias, 0};
    }
  } else {
    // Pool staging is small: the warpgroups always take alternate tiles.
    const int gmin = mode == MODE_POOL ? 2 : 1;
    for (int resident = 1; resident >= 0; --resident)
      for (int groups = 2; groups >= gmin; --groups) cands[ncand++] = {2, groups, resident, 0, 0};
  }

  int feas[16];
  uint32_t feas_stages[16], feas_stage_bytes[16];
  int nfeas = 0;
  {
    for (int c = 0; c < ncand; ++c) {
      const Cand& k = cands[c];
      // Resident filters of an R > 1 conv: one halo box of (8 + R - 1) x 16 pixels per
      // column tap and channel block feeds all R row taps.
      const uint32_t a_bytes = (k.resident && p.R > 1 && p.stride == 1)
                                   ? (7u + static_cast<uint32_t>(p.R)) * 2048u
                                   : kABytes;
      const uint32_t stage_bytes =
          k.resident ? a_bytes
          : k.w0res  ? round_up(std::max(kABytes, p.w1_chunk_bytes), 1024u)
                     : round_up(std::max(kABytes + p.w0_chunk_bytes, p.w1_chunk_bytes), 1024u);
      const uint32_t pbufs = (mode == MODE_CHAIN && !k.p_tmem) ? static_cast<uint32_t>(k.dual) : 0u;
      const uint32_t obufs = k.w0res ? 0u : (k.groups == 2 && !k.two ? 2u : 1u);
      const uint32_t shared = k.alias ? pbufs * std::max(p_bytes, out_bytes)
                                      : pbufs * p_bytes + obufs * (k.two ? slot_bytes : out_bytes);
      const uint32_t w0_res_bytes = static_cast<uint32_t>(p.kchunks0) * p.w0_chunk_bytes;
      const uint32_t fixed =
          (k.resident ? w_res : k.w0res ? w0_res_bytes : 0u) + shared + bias_bytes + bar_bytes;
      if (fixed >= budget) continue;
      const uint32_t stages = std::min<uint32_t>(kMaxStages, (budget - fixed) / stage_bytes);
      if (stages < 2u) continue;
      if (k.two && stages / 2u < static_cast<uint32_t>(p.S * p.kc_per_tap)) continue;
      feas[nfeas] = c;
      feas_stages[nfeas] = stages;
      feas_stage_bytes[nfeas++] = stage_bytes;
    }
  }
  int pick = -1;
  if (forced >= 0) {
    pick = forced < nfeas ? forced : -1;
  } else {
    for (int i = 0; i < nfeas && pick < 0; ++i)
      if (feas_stages[i] >= 3u) pick = i;
    if (pick < 0 && nfeas > 0) pick = 0;
  }
  if (pick < 0) return false;
  const int chosen = feas[pick];
  const uint32_t chosen_stages = feas_stages[pick], chosen_stage_bytes = feas_stage_bytes[pick];
  const Cand& k = cands[chosen];
  p.acc_dual = k.dual >= 2 ? 1 : 0;
  p.nbuf_log2 = mode != MODE_CHAIN ? 1 : (k.dual == 4 ? 2 : (k.dual == 2 ? 1 : 0));
  p.epi_groups = k.groups;
  p.resident = k.resident;
  p.w0_res = k.w0res;
  p.out_alias_p = k.alias;
  p.p_tmem = k.p_tmem;
  p.num_stages = chosen_stages;
  p.stage_bytes = chosen_stage_bytes;
  p.halo = (k.resident && p.R > 1 && p.stride == 1) ? 1 : 0;
  p.a_stage_bytes = p.halo ? (7u + static_cast<uint32_t>(p.R)) * 2048u : kABytes;
  p.kstages0 = p.halo ? p.S * p.kc_per_tap : p.kchunks0;
  p.two_issuers = k.two;
  p.out_slots = k.two;
  p.tmem_cols = tmem_layout(p, mode, static_cast<uint32_t>(k.dual), k.p_tmem != 0);
  // P in TMEM with streamed weights: W1 is packed into as few ring stages as possible and
  // shared by the two tiles of a pair -- if those stages fit the ring at once.
  p.w1_group = 0;
  p.w1_per_stage = 1;
  if (mode == MODE_CHAIN && k.p_tmem && !k.resident && p.p_split == 0u) {
    const uint32_t per = std::max(1u, p.stage_bytes / p.w1_chunk_bytes);
    const uint32_t stages = (static_cast<uint32_t>(p.kchunks1) + per - 1) / per;
    if (stages <= p.num_stages) {
      p.w1_group = 1;
      p.w1_per_stage = per;
    }
  }
  // Wide chains (one tile in flight): W1 packed the same way for every tile, so that its
  // GEMM1 waits for two ring fills instead of one per chunk.
  if (mode == MODE_CHAIN && !k.resident && p.p_split != 0u)
    p.w1_per_stage = std::max(1u, p.stage_bytes / p.w1_chunk_bytes);
  // The conv + pool kernel with N <= 64: two MMA issuers over two sub-rings, each holding
  // all the ring stages of one tile (measured, N = 64, three stages per tile in a
  // seven-stage ring: 39.4 -> 35.6 us).  With longer MMAs one issuer keeps the tensor core
  // busy, and sub-rings shallower than a tile starve both issuers; on the single GEMMs of
  // the unfused operators (also tried: N = 64 and N = 128-256) two issuers ran 2-10 %
  // slower, so they keep one.
  if (mode == MODE_POOL)
    p.two_issuers =
        p.N0p <= 64 && p.num_stages / 2u >= static_cast<uint32_t>(p.kstages0) ? 1 : 0;
  // ... and each issuer two accumulators, so that it starts its next tile while the
  // epilogue drains the previous one (tile i takes buffer i & 3)
  if (mode == MODE_POOL && p.two_issuers && tmem_layout(p, mode, 4u) <= 512u) {
    p.nbuf_log2 = 2;
    p.tmem_cols = tmem_layout(p, mode, 4u);
  } else {
    p.tmem_cols = tmem_layout(p, mode, static_cast<uint32_t>(k.dual), k.p_tmem != 0);
  }
  Regions r;
  r.cand = pick;
  r.ncand = nfeas;
  r.ring = p.num_stages * p.stage_bytes;
  r.w_res = p.resident ? w_res : (k.w0res ? static_cast<uint32_t>(p.kchunks0) * p.w0_chunk_bytes : 0u);
  const uint32_t pbufs = (mode == MODE_CHAIN && !k.p_tmem) ? static_cast<uint32_t>(k.dual) : 0u;
  r.p_each = pbufs ? (p.out_alias_p ? std::max(p_bytes, out_bytes) : p_bytes) : 0u;
  r.out_each = (p.out_alias_p || k.w0res) ? 0u : (k.two ? slot_bytes : out_bytes);
  r.bias = bias_bytes;
  r.bar = bar_bytes;
  const uint32_t obufs = k.w0res ? 0u : (k.groups == 2 && !k.two ? 2u : 1u);
  uint32_t off = 0;
  p.off_ring = off;
  off += r.ring;
  p.off_w0 = off;
  p.off_w1 = off + static_cast<uint32_t>(p.kchunks0) * p.w0_chunk_bytes;
  off += r.w_res;
  for (uint32_t b = 0; b < kMaxBufs; ++b) p.off_p[b] = off + (b < pbufs ? b : 0u) * r.p_each;
  off += pbufs * r.p_each;
  for (uint32_t b = 0; b < 2; ++b) {
    if (p.out_alias_p) p.off_out[b] = p.off_p[b];
    else if (obufs == 0u) p.off_out[b] = 0u;   // no staging (never read)
    else p.off_out[b] = off + (b < obufs ? b : 0u) * r.out_each;
  }
  if (!p.out_alias_p) off += obufs * r.out_each;
  p.off_bias = off;
  off += r.bias;
  p.off_bar = off;
  off += r.bar;
  // When the output staging directly follows the ring (streamed weights, P in TMEM) and W1
  // is loaded once per tile pair, a CTA with at most two tiles never fills the ring after
  // its second tile's GEMM0 except with W1, so stages that run on into the staging are
  // free before any epilogue writes it (the epilogue waits for GEMM1, which follows every
  // GEMM0 chunk).  The extra stages are counted here and taken at launch when the grid
  // gives no CTA a third tile, provided that W1's stages of the pair miss them.
  r.extend = 0;
  if (mode == MODE_CHAIN && k.p_tmem && !k.resident && !k.w0res && p.w1_group &&
      p.off_out[0] == p.off_ring + r.ring) {
    const uint32_t span = r.ring + obufs * r.out_each;
    const uint32_t total = std::min<uint32_t>(kMaxStages, span / p.stage_bytes);
    const uint32_t w1_stages = (static_cast<uint32_t>(p.kchunks1) + p.w1_per_stage - 1) /
                               p.w1_per_stage;
    bool clear = total > p.num_stages;
    for (uint32_t j = 0; j < w1_stages && clear; ++j)
      clear = (2u * static_cast<uint32_t>(p.kstages0) + j) % total < p.num_stages;
    if (clear) r.extend = total - p.num_stages;
  }
  *smem_bytes = off + 1024u;
  if (regions) *regions = r;
  return *smem_bytes <= kSmemLimit && p.tmem_cols <= 512u;
}

// Shared-memory plan of the three-operator chain: ring of A chunks; W0, W1, W2 resident
// (W2 written by the epilogue warps in the same MN-major layout as a TMA load of W1);
// two P0, two P1 and two output staging buffers (tile i uses buffer i & 1); bias operands
// of the three GEMMs; barriers.  At least two ring stages, else the chain does not fit.
bool plan_smem_chain3(ChainParams& p, size_t* smem_bytes, Regions* regions) {
  const uint32_t budget = kSmemLimit - 1024u;
  const uint32_t n0blk = static_cast<uint32_t>((p.N0p + 63) / 64);
  const uint32_t n1blk = static_cast<uint32_t>((p.N1p + 63) / 64);
  const uint32_t n2blk = static_cast<uint32_t>((p.N2p + 63) / 64);
  p.w0_chunk_bytes = n0blk * 8192u;
  p.w1_chunk_bytes = n1blk * 8192u;
  p.w2_chunk_bytes = n2blk * 8192u;
  const uint32_t p0_bytes = n0blk * kPChunkBytes, p1_bytes = n1blk * kPChunkBytes;
  const uint32_t out_bytes = n2blk * kPChunkBytes;
  const uint32_t bias_bytes = kOnesBytes + kBiasBlockBytes * (n0blk + n1blk + n2blk);
  const uint32_t bar_bytes = 1024u;
  const uint32_t w_res = static_cast<uint32_t>(p.kchunks0) * p.w0_chunk_bytes +
                         static_cast<uint32_t>(p.kchunks1) * p.w1_chunk_bytes +
                         static_cast<uint32_t>(p.kchunks2) * p.w2_chunk_bytes;
  // The output staging of buffer b may share P0[b]'s space: the group that owns buffer b
  // writes it only after GEMM2 of the tile (so GEMM1 has read P0[b]) and waits for the TMA
  // store to have read it before its next tile's P0.  Taken when separate staging would
  // leave fewer than three ring stages.
  auto stages_for = [&](bool alias) -> uint32_t {
    const uint64_t fixed = uint64_t{w_res} +
                           2u * ((alias ? std::max(p0_bytes, out_bytes) : p0_bytes + out_bytes) +
                                 p1_bytes) +
                           bias_bytes + bar_bytes;
    if (fixed >= budget) return 0u;
    return std::min<uint32_t>(kMaxStages, (budget - static_cast<uint32_t>(fixed)) / kABytes);
  };
  const bool alias = stages_for(false) < 3u && stages_for(true) > stages_for(false);
  const uint32_t stages = stages_for(alias);
  if (stages < 2u) return false;
  const uint32_t p0_each = alias ? std::max(p0_bytes, out_bytes) : p0_bytes;
  p.tmem_cols = tmem_layout(p, MODE_CHAIN3, 2u);
  if (p.tmem_cols > 512u) return false;
  p.acc_dual = 1;
  p.nbuf_log2 = 1;
  p.epi_groups = 2;
  p.resident = 1;
  p.out_alias_p = alias ? 1 : 0;
  p.p_tmem = 0;
  p.halo = 0;
  p.num_stages = stages;
  p.stage_bytes = kABytes;
  p.a_stage_bytes = kABytes;
  p.kstages0 = p.kchunks0;
  p.w1_group = 0;
  p.w1_per_stage = 1;
  Regions r;
  r.cand = 0;
  r.ncand = 1;
  r.ring = stages * kABytes;
  r.w_res = w_res;
  r.p_each = p0_each;
  r.out_each = alias ? 0u : out_bytes;
  r.bias = bias_bytes;
  r.bar = bar_bytes;
  uint32_t off = 0;
  p.off_ring = off;
  off += r.ring;
  p.off_w0 = off;
  p.off_w1 = p.off_w0 + static_cast<uint32_t>(p.kchunks0) * p.w0_chunk_bytes;
  p.off_w2 = p.off_w1 + static_cast<uint32_t>(p.kchunks1) * p.w1_chunk_bytes;
  off += w_res;
  for (uint32_t b = 0; b < kMaxBufs; ++b) p.off_p[b] = off + (b & 1u) * p0_each;
  off += 2u * p0_each;
  for (uint32_t b = 0; b < 2; ++b) p.off_p1[b] = off + b * p1_bytes;
  off += 2u * p1_bytes;
  for (uint32_t b = 0; b < 2; ++b) p.off_out[b] = alias ? p.off_p[b] : off + b * out_bytes;
  if (!alias) off += 2u * out_bytes;
  p.off_bias = off;
  off += bias_bytes;
  p.off_bar = off;
  off += bar_bytes;
  *smem_bytes = off + 1024u;
  if (regions) *regions = r;
  return *smem_bytes <= kSmemLimit;
}

// The CTA-pair plan of a b2b GEMM chain with row-major weights (chain_cta2_kernel.cuh): per
// CTA a ring of 16 KiB A chunks, its halves of W0 and W1 resident (N0 / 2 and N1 / 2
// columns), the bias operands of its halves and the barriers (no output staging: the
// epilogue stores the output from registers); in TMEM the tile-pair layout with P kept over GEMM0's
// columns.  p.num_tiles becomes the number of 256-row tiles.
// False when the chain is outside the kernel's limits (N0 or N1 not a multiple of 128,
// more than kMaxW0Chunks K chunks, the TMEM layout over 512 columns, fewer than three ring
// stages beside the weights).
constexpr uint32_t kCta2StagingBytes = 8u * 4096u;   // 32 rows x 64 columns per epilogue warp

bool plan_cta2(ChainParams& p, size_t* smem_bytes, Regions* regions) {
  if (p.N0p % 128 != 0 || p.N1p % 128 != 0 || p.N0p > 256 || p.N1p > 256) return false;
  if (p.kchunks0 > kMaxW0Chunks || p.kchunks0 < 1) return false;
  const uint32_t budget = kSmemLimit - 1024u;
  const uint32_t nb0 = static_cast<uint32_t>(p.N0p / 128), nb1 = static_cast<uint32_t>(p.N1p / 128);
  p.w0_chunk_bytes = nb0 * 8192u;
  p.w1_chunk_bytes = nb1 * 8192u;
  const uint32_t w0b = static_cast<uint32_t>(p.kchunks0) * p.w0_chunk_bytes;
  const uint32_t w1b = static_cast<uint32_t>(p.kchunks1) * p.w1_chunk_bytes;
  const uint32_t bias_bytes = kOnesBytes + kBiasBlockBytes * (nb0 + nb1);
  const uint32_t bar_bytes = 1024u;
  const uint32_t fixed = w0b + w1b + bias_bytes + bar_bytes;
  if (fixed >= budget) return false;
  // The output leaves through a 4 KiB staging slot per epilogue warp and TMA stores when
  // the ring keeps five stages beside it (measured on the FFN-like chain: five stages run
  // as fast as seven, four do not); else from registers.
  const bool stage_out = fixed + kCta2StagingBytes < budget &&
                         (budget - fixed - kCta2StagingBytes) / kABytes >= 5u;
  const uint32_t staging = stage_out ? kCta2StagingBytes : 0u;
  const uint32_t stages = std::min<uint32_t>(kMaxStages, (budget - fixed - staging) / kABytes);
  if (stages < 3u) return false;
  p.tmem_cols = tmem_layout(p, MODE_CHAIN, 2u, true);
  if (p.tmem_cols > 512u) return false;
  p.cta_pair = 1;
  p.num_tiles = ceil_div(p.M, 2 * kBlockM);
  p.acc_dual = 1;
  p.nbuf_log2 = 1;
  p.epi_groups = 2;
  p.resident = 1;
  p.w0_res = 0;
  p.out_alias_p = 0;
  p.p_tmem = 1;
  p.halo = 0;
  p.num_stages = stages;
  p.stage_bytes = kABytes;
  p.a_stage_bytes = kABytes;
  p.kstages0 = p.kchunks0;
  p.w1_group = 0;
  p.w1_per_stage = 1;
  uint32_t off = 0;
  p.off_ring = off;
  off += stages * kABytes;
  p.off_w0 = off;
  p.off_w1 = off + w0b;
  off += w0b + w1b;
  for (uint32_t b = 0; b < kMaxBufs; ++b) p.off_p[b] = 0;
  p.off_out[0] = p.off_out[1] = 0;
  p.out_stage = stage_out ? 1 : 0;
  if (stage_out) {
    p.off_out[0] = off;
    off += staging;
  }
  p.off_bias = off;
  off += bias_bytes;
  p.off_bar = off;
  off += bar_bytes;
  if (regions) {
    Regions r;
    r.ring = stages * kABytes;
    r.w_res = w0b + w1b;
    r.p_each = 0;
    r.out_each = staging;
    r.bias = bias_bytes;
    r.bar = bar_bytes;
    *regions = r;
  }
  *smem_bytes = off + 1024u;
  return *smem_bytes <= kSmemLimit;
}

// Shared-memory plan of the conv + pool kernel over CTA pairs (chain_cta2_pool_kernel.cuh;
// stride 1, R > 1, N0p <= 128): per CTA a ring of halo boxes of its own 8 x 16 tile, its
// half of the filters resident (N0p / 2 rows of every tap and channel block), one pooled
// staging tile per epilogue warpgroup, the bias of every channel (fp32), the barriers; two
// accumulators of N0p columns in TMEM per MMA issuer.  At least one tile's ring stages
// and one more.  p.num_tiles stays the count of 8 x 16 tiles (two per pair-tile).
bool plan_pool_cta2(ChainParams& p, size_t* smem_bytes, Regions* regions) {
  if (p.R < 2 || p.stride != 1 || p.N0p > 128 || p.N0p % 16 != 0) return false;
  const uint32_t budget = kSmemLimit - 1024u;
  const uint32_t half = static_cast<uint32_t>(p.N0p) / 2u;
  p.w0_chunk_bytes = half * 128u;
  const uint32_t w0b = static_cast<uint32_t>(p.kchunks0) * p.w0_chunk_bytes;
  const uint32_t nch = static_cast<uint32_t>((p.N0p + 63) / 64);
  const uint32_t out_each = nch * kPoolChunkBytes;
  const uint32_t bias_bytes = 1024u;   // 256 fp32 words: the bias of every channel
  const uint32_t bar_bytes = 1024u;
  const uint32_t a_bytes = (7u + static_cast<uint32_t>(p.R)) * 2048u;
  const uint32_t kst = static_cast<uint32_t>(p.S * p.kc_per_tap);
  const uint32_t fixed = round_up(w0b, 1024u) + 2u * out_each + bias_bytes + bar_bytes;
  if (fixed >= budget) return false;
  const uint32_t stages = std::min<uint32_t>(kPool2MaxStages, (budget - fixed) / a_bytes);
  if (stages < kst + 1u) return false;
  const uint32_t s0 = round_up(static_cast<uint32_t>(p.N0p), 32u);
  // MMA issuers in the leader, each over a sub-ring that holds a tile's stages, each with
  // two accumulator buffers: three where six buffers fit TMEM, else two, else one
  uint32_t issuers = std::min<uint32_t>(3u, stages / kst);
  if (issuers == 3u && 6u * s0 > 512u) issuers = 2u;
  if (issuers == 0u) issuers = 1u;
  p.tmem_cols = pow2_at_least((issuers == 3u ? 6u : 4u) * s0);
  if (p.tmem_cols > 512u) return false;
  for (uint32_t b = 0; b < kMaxBufs; ++b) {
    p.d0_col[b] = b * s0;
    p.d1_col[b] = 0;
  }
  p.cta_pair = 1;
  p.acc_dual = 1;
  p.nbuf_log2 = 2;
  p.epi_groups = 2;
  p.resident = 1;
  p.w0_res = 0;
  p.out_alias_p = 0;
  p.p_tmem = 0;
  p.halo = 1;
  p.two_issuers = static_cast<int32_t>(issuers) - 1;
  p.num_stages = stages;
  p.stage_bytes = a_bytes;
  p.a_stage_bytes = a_bytes;
  p.kstages0 = static_cast<int32_t>(kst);
  p.w1_group = 0;
  p.w1_per_stage = 1;
  uint32_t off = 0;
  p.off_ring = off;
  off += stages * a_bytes;
  p.off_w0 = off;
  p.off_w1 = off;
  off += round_up(w0b, 1024u);
  for (uint32_t b = 0; b < kMaxBufs; ++b) p.off_p[b] = 0;
  p.off_out[0] = off;
  p.off_out[1] = off + out_each;
  off += 2u * out_each;
  p.off_bias = off;
  off += bias_bytes;
  p.off_bar = off;
  off += bar_bytes;
  if (regions) {
    Regions r;
    r.ring = stages * a_bytes;
    r.w_res = round_up(w0b, 1024u);
    r.p_each = 0;
    r.out_each = out_each;
    r.bias = bias_bytes;
    r.bar = bar_bytes;
    *regions = r;
  }
  *smem_bytes = off + 1024u;
  return *smem_bytes <= kSmemLimit;
}

void fill_common(ChainParams& p, int dt, int e0, int e1, const void* b0, const void* b1,
                 DeviceState* d, uint32_t kid) {
  p.is_bf16 = dt == B2B_BF16 ? 1 : 0;
  p.act0 = e0;
  p.act1 = e1;
  p.b0 = static_cast<const uint16_t*>(b0);
  p.b1 = static_cast<const uint16_t*>(b1);
  p.wait_limit_ns = g_wait_ns.load();
  p.kernel_id = kid;
  p.err = d ? d->err : nullptr;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  p.trace = g_trace_buf;
  p.trace_cap = g_trace_cap;
  p.trace_cta = g_trace_cta;
}

// Lets the kernel of variant v (the launch's dtype and build) use the full shared memory.
b2b_status ensure_smem_attribute(Variant v, DeviceState* d, bool bf16, bool traced) {
  const uint32_t idx = 2u * (static_cast<uint32_t>(v) + (traced ? V_COUNT : 0u)) + (bf16 ? 1u : 0u);
  static_assert(4 * V_COUNT <= 128, "attribute bits");
  std::atomic<uint64_t>& word = d->attr_done[idx >> 6];
  const uint64_t bit = 1ull << (idx & 63u);
  if ((word.load() & bit) == 0u) {
    if (cudaFuncSetAttribute(variant_func(v, bf16, traced),
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemLimit)) != cudaSuccess) {
      cudaGetLastError();
      return B2B_ERR_CUDA;
    }
    word.fetch_or(bit);
  }
  return B2B_OK;
}

b2b_status launch(Variant v, DeviceState* d, const CUtensorMap& a, const CUtensorMap& w0,
                  const CUtensorMap& w1, const CUtensorMap& out, ChainParams& p, size_t smem,
                  int grid, void* stream) {
  const bool traced = p.trace != nullptr;
  if (b2b_status st = ensure_smem_attribute(v, d, p.is_bf16 != 0, traced); st != B2B_OK)
    return st;
  const cudaError_t e =
      launch_variant(v, a, w0, w1, out, p, grid, smem, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return B2B_ERR_CUDA;
  }
  return B2B_OK;
}

// ------------------------------------------------------------------------------------
// launch parameters (host only; no CUDA call)
// ------------------------------------------------------------------------------------
// 2-D A operand.  W0/W1 are [K][N] row-major when w_mn, else [N][K] (conv filters).
bool gemm_params(ChainParams& p, int mode, bool w_mn, int64_t M, int32_t K0, int32_t N0,
                 int32_t N1, size_t* smem, Regions* regions, int forced = -1) {
  std::memset(&p, 0, sizeof(p));
  p.M = static_cast<int32_t>(M);
  p.K0 = K0;
  p.N0 = N0;
  p.N1 = mode == MODE_CHAIN ? N1 : 0;
  p.N0p = static_cast<int32_t>(round_up(static_cast<uint32_t>(N0), 16u));
  p.N1p = mode == MODE_CHAIN ? static_cast<int32_t>(round_up(static_cast<uint32_t>(N1), 16u)) : 0;
  p.kchunks0 = ceil_div(K0, kChunkK);
  p.kc_per_tap = p.kchunks0;
  p.kchunks1 = mode == MODE_CHAIN ? ceil_div(p.N0p, kChunkK) : 0;
  p.num_tiles = ceil_div(M, kBlockM);
  p.stride = 1;
  // A chain with row-major weights may also run over CTA pairs: that plan is one more
  // feasible layout, after the single-CTA ones (last in the order of preference; the
  // tile-graph model takes it where its bounds are lower and every pair runs three or
  // more tiles -- measured on the FFN-like chain: 12.0 against 13.1 us at 40000 rows,
  // 44.6 against 53.0 us at 262144, but 9.8 against 9.3 us at 32768, two tiles per pair,
  // where the pairs' longer start is not amortised).
  if (mode == MODE_CHAIN && w_mn) {
    ChainParams q = p;
    size_t qs = 0;
    Regions qr;
    const bool single_ok = plan_smem(q, mode, true, true, &qs, &qr, -1);
    const int nsingle = single_ok ? qr.ncand : 0;
    ChainParams c = p;
    size_t cs = 0;
    Regions cr;
    const bool pair_ok = plan_cta2(c, &cs, &cr);
    if (pair_ok && forced == nsingle) {
      p = c;
      *smem = cs;
      if (regions) {
        *regions = cr;
        regions->cand = nsingle;
        regions->ncand = nsingle + 1;
      }
      return true;
    }
    const bool ok = plan_smem(p, mode, w_mn, w_mn, smem, regions, forced);
    if (ok && pair_ok && regions) regions->ncand += 1;
    return ok;
  }
  return plan_smem(p, mode, w_mn, w_mn, smem, regions, forced);
}

// Three-operator chain over a 2-D A with row-major W0 [K0][N0], W1 [N0][N1], W2 [N1][N2].
bool gemm3_params(ChainParams& p, int64_t M, int32_t K0, int32_t N0, int32_t N1, int32_t N2,
                  size_t* smem, Regions* regions, int forced = -1) {
  std::memset(&p, 0, sizeof(p));
  if (forced > 0) return false;   // one layout
  p.M = static_cast<int32_t>(M);
  p.K0 = K0;
  p.N0 = N0;
  p.N1 = N1;
  p.N2 = N2;
  p.N0p = static_cast<int32_t>(round_up(static_cast<uint32_t>(N0), 16u));
  p.N1p = static_cast<int32_t>(round_up(static_cast<uint32_t>(N1), 16u));
  p.N2p = static_cast<int32_t>(round_up(static_cast<uint32_t>(N2), 16u));
  p.kchunks0 = ceil_div(K0, kChunkK);
  p.kc_per_tap = p.kchunks0;
  p.kchunks1 = ceil_div(p.N0p, kChunkK);
  p.kchunks2 = ceil_div(p.N1p, kChunkK);
  p.num_tiles = ceil_div(M, kBlockM);
  p.stride = 1;
  return plan_smem_chain3(p, smem, regions);
}

// 4-D implicit-GEMM A operand (conv filters [Cout][R][S][Cin]).
bool conv_params(ChainParams& p, int mode, int32_t N, int32_t H, int32_t W, int32_t C,
                 int32_t C0, int32_t R, int32_t S, int32_t pad, int32_t C1, size_t* smem,
                 Regions* regions, int forced = -1, int32_t stride = 1) {
  std::memset(&p, 0, sizeof(p));
  p.K0 = C;
  p.N0 = C0;
  p.N1 = mode == MODE_CHAIN ? C1 : 0;
  p.N0p = static_cast<int32_t>(round_up(static_cast<uint32_t>(C0), 16u));
  p.N1p = mode == MODE_CHAIN ? static_cast<int32_t>(round_up(static_cast<uint32_t>(C1), 16u)) : 0;
  p.kc_per_tap = ceil_div(C, kChunkK);
  p.kchunks0 = R * S * p.kc_per_tap;
  p.kchunks1 = mode == MODE_CHAIN ? ceil_div(p.N0p, kChunkK) : 0;
  p.R = R;
  p.S = S;
  p.pad = pad;
  p.stride = stride;
  p.Ho = (H + 2 * pad - R) / stride + 1;
  p.Wo = (W + 2 * pad - S) / stride + 1;
  p.tiles_w = ceil_div(p.Wo, 16);
  p.tiles_h = ceil_div(p.Ho, 8);
  const int64_t tiles = static_cast<int64_t>(N) * p.tiles_w * p.tiles_h;
  if (tiles > INT32_MAX) return false;
  p.num_tiles = static_cast<int32_t>(tiles);
  // The conv + pool may also run over CTA pairs: one more feasible layout after the
  // single-CTA ones (as for the b2b GEMM chain).
  if (mode == MODE_POOL) {
    ChainParams q = p;
    size_t qs = 0;
    Regions qr;
    const bool single_ok = plan_smem(q, mode, false, false, &qs, &qr, -1);
    const int nsingle = single_ok ? qr.ncand : 0;
    ChainParams c = p;
    size_t cs = 0;
    Regions cr;
    const bool pair_ok = plan_pool_cta2(c, &cs, &cr);
    if (pair_ok && forced == nsingle) {
      p = c;
      *smem = cs;
      if (regions) {
        *regions = cr;
        regions->cand = nsingle;
        regions->ncand = nsingle + 1;
      }
      return true;
    }
    const bool ok = plan_smem(p, mode, false, false, smem, regions, forced);
    if (ok && pair_ok && regions) regions->ncand += 1;
    return ok;
  }
  return plan_smem(p, mode, false, false, smem, regions, forced);
}

// ------------------------------------------------------------------------------------
// launch choices
// ------------------------------------------------------------------------------------
// What a launch of one problem may vary without changing its results (the same MMAs in
// the same order, the same roundings): the shared-memory / TMEM layout (an index into the
// planner's feasible candidates), the grid (0: one CTA per SM, or per tile if fewer;
// 1: the fewest CTAs that keep the busiest CTA's tile count; 2: one CTA per tile, in
// waves) and whether each CTA's second tile's A rows are prefetched into L2 at the start.
// -1 leaves a field to the planner's default.
struct Choice {
  int32_t cand = -1, grid = -1, pf2 = -1;
};

// What one launch looked like, for the profiler's enumeration.
constexpr int kGridModes = 3;
struct Info {
  int32_t cand = 0;   // the layout the launch took (the planner's default when not forced)
  int32_t ncand = 0, tiles = 0, can_prefetch = 0;
  int32_t grid[kGridModes] = {0, 0, 0};   // the grid of each mode
};

int grid_for(int32_t tiles, int sms, int32_t mode) {
  const int full = std::max(1, std::min<int>(tiles, sms));
  if (mode == 2) return std::max(1, tiles);
  if (mode != 1) return full;
  const int per = (tiles + full - 1) / full;
  return std::max(1, (tiles + per - 1) / per);
}

Info info_for(const Regions& r, int32_t tiles, int sms, bool can_prefetch) {
  Info i;
  i.cand = r.cand;
  i.ncand = r.ncand;
  i.tiles = tiles;
  i.can_prefetch = can_prefetch ? 1 : 0;
  for (int m = 0; m < kGridModes; ++m) i.grid[m] = grid_for(tiles, sms, m);
  return i;
}

// Default: prefetch the second tile too when a CTA has more than two tiles -- then the
// rolling prefetch (two tiles ahead) starts from the third; with one or two tiles per
// CTA the second tile's prefetch competed with the first tile's loads (measured on the
// FFN-shaped chain: 1 % slower with it).
int32_t pf_second_for(int32_t tiles, int grid, int32_t pf2) {
  if (pf2 >= 0) return pf2 != 0 ? 1 : 0;
  return (tiles + grid - 1) / grid > 2 ? 1 : 0;
}

// ------------------------------------------------------------------------------------
// GEMM-shaped entry points (2-D A operand)
// ------------------------------------------------------------------------------------
// The b2b GEMM chain over CTA pairs (plan_cta2): clusters of two CTAs, at most as many as
// can be resident at once; grid choices as for single CTAs, counted in pairs.
b2b_status run_cta2(const Choice& ch, Info* info, const Regions& r, ChainParams& p, size_t smem,
                    DeviceState* d, int dt, int64_t M, int32_t K0, int32_t N0, int32_t N1,
                    const void* A, const void* W0, const void* b0, int e0, const void* W1,
                    const void* b1, int e1, void* D, void* stream) {
  fill_common(p, dt, e0, e1, b0, b1, d, KID_GEMM_CHAIN_CTA2);
  const bool traced = p.trace != nullptr;
  if (b2b_status st = ensure_smem_attribute(V_GEMM_CHAIN_CTA2, d, p.is_bf16 != 0, traced);
      st != B2B_OK)
    return st;
  const int ci = (p.is_bf16 ? 1 : 0) + (traced ? 2 : 0);
  int clusters = d->cta2_clusters[ci].load();
  if (clusters <= 0 || d->cta2_smem[ci].load() != smem) {
    if (cta2_max_clusters(p.is_bf16 != 0, traced, smem, &clusters) != cudaSuccess || clusters < 1) {
      cudaGetLastError();
      return B2B_ERR_CUDA;
    }
    d->cta2_clusters[ci].store(clusters);
    d->cta2_smem[ci].store(smem);
  }
  const int pairs = grid_for(p.num_tiles, clusters, ch.grid);
  p.pf_second = 0;
  if (info) *info = info_for(r, p.num_tiles, clusters, true);
  const uint64_t e = 2;
  CUtensorMap ta, tw0, tw1;
  bool ok = make_map(&ta, A, p.is_bf16, 2, {static_cast<uint64_t>(K0), static_cast<uint64_t>(M)},
                     {K0 * e}, {kChunkK, kBlockM});
  // [N/64][rows][64] views of the row-major weights; each CTA loads its half of the
  // 64-wide blocks of every K chunk in one box
  ok = ok && make_map(&tw0, W0, p.is_bf16, 3,
                      {64, static_cast<uint64_t>(K0), static_cast<uint64_t>(N0 / 64)}, {N0 * e, 128},
                      {64, 64, static_cast<uint32_t>(p.N0p / 128)});
  ok = ok && make_map(&tw1, W1, p.is_bf16, 3,
                      {64, static_cast<uint64_t>(N0), static_cast<uint64_t>(N1 / 64)}, {N1 * e, 128},
                      {64, 64, static_cast<uint32_t>(p.N1p / 128)});
  if (!ok) return B2B_ERR_CUDA;
  p.pf_a = static_cast<const uint8_t*>(A);
  p.pf_a_bytes = static_cast<uint64_t>(M) * K0 * e;
  p.pf_a_tile_bytes = static_cast<uint32_t>(kBlockM * K0 * e);
  p.out_ptr = static_cast<uint8_t*>(D);
  p.out_ld = N1;
  // The output map stores one warp's 32 rows x 64 columns per box (staged output only).
  CUtensorMap to = ta;
  if (p.out_stage &&
      !make_map(&to, D, p.is_bf16, 2, {static_cast<uint64_t>(N1), static_cast<uint64_t>(M)},
                {N1 * e}, {64, 32}))
    return B2B_ERR_CUDA;
  return launch(V_GEMM_CHAIN_CTA2, d, ta, tw0, tw1, to, p, smem, 2 * pairs, stream);
}

b2b_status run_gemm_with(const Choice& ch, Info* info, int mode, bool w_mn, int dt, int64_t M,
                         int32_t K0, int32_t N0, int32_t N1, const void* A, const void* W0,
                         const void* b0, int e0, const void* W1, const void* b1, int e1, void* D,
                         void* stream, uint32_t kid) {
  ChainParams p;
  size_t smem = 0;
  Regions r;
  if (!gemm_params(p, mode, w_mn, M, K0, N0, N1, &smem, &r, ch.cand)) return B2B_ERR_UNSUPPORTED;
  b2b_status st = B2B_OK;
  DeviceState* d = device_state(&st);
  if (d == nullptr) return st;
  if (p.cta_pair)
    return run_cta2(ch, info, r, p, smem, d, dt, M, K0, N0, N1, A, W0, b0, e0, W1, b1, e1, D,
                    stream);
  fill_common(p, dt, e0, e1, b0, b1, d, kid);
  const int grid = grid_for(p.num_tiles, d->num_sms, ch.grid);
  p.pf_second = pf_second_for(p.num_tiles, grid, ch.pf2);
  if (r.extend > 0 && (p.num_tiles + grid - 1) / grid <= 2) p.num_stages += r.extend;
  if (info) *info = info_for(r, p.num_tiles, d->num_sms, true);

  CUtensorMap ta, tw0, tw1, to;
  const uint64_t e = 2;
  bool ok = make_map(&ta, A, p.is_bf16, 2, {static_cast<uint64_t>(K0), static_cast<uint64_t>(M)},
                     {K0 * e}, {kChunkK, kBlockM});
  // A row-major [rows][N] tensor with N a multiple of 64 viewed as [N/64][rows][64]: one
  // box then covers every 64-wide column block of `box_rows` rows, laid out block after
  // block exactly as the kernel's per-block boxes land.  Returns false (and the caller
  // keeps the per-block 2-D map) if N is ragged or the driver refuses the view.
  // A box of `box_blocks` blocks (all of them by default).
  auto map3 = [&](CUtensorMap* m, const void* ptr, uint64_t rows, int32_t N, uint32_t box_rows,
                  uint32_t box_blocks = 0) {
    if (N % 64 != 0) return false;
    const uint32_t nb = static_cast<uint32_t>(N / 64);
    return make_map(m, ptr, p.is_bf16, 3, {64, rows, nb}, {N * e, 128},
                    {64, box_rows, box_blocks ? std::min(box_blocks, nb) : nb});
  };
  if (w_mn) {
    // Wide chains load W0 by halves of N0: boxes of four blocks.
    p.w0_box3 = map3(&tw0, W0, static_cast<uint64_t>(K0), N0, 64, p.p_split ? 4u : 0u) ? 1 : 0;
    if (!p.w0_box3)
      ok = ok && make_map(&tw0, W0, p.is_bf16, 2,
                          {static_cast<uint64_t>(N0), static_cast<uint64_t>(K0)}, {N0 * e}, {64, 64});
  } else
    ok = ok && make_map(&tw0, W0, p.is_bf16, 2, {static_cast<uint64_t>(K0), static_cast<uint64_t>(N0)},
                        {K0 * e}, {kChunkK, static_cast<uint32_t>(p.N0p)});
  const int32_t Nout = mode == MODE_CHAIN ? N1 : N0;
  if (mode == MODE_CHAIN) {
    if (w_mn) {
      p.w1_box3 = map3(&tw1, W1, static_cast<uint64_t>(N0), N1, 64) ? 1 : 0;
      if (!p.w1_box3)
        ok = ok && make_map(&tw1, W1, p.is_bf16, 2,
                            {static_cast<uint64_t>(N1), static_cast<uint64_t>(N0)}, {N1 * e}, {64, 64});
    } else
      ok = ok && make_map(&tw1, W1, p.is_bf16, 2, {static_cast<uint64_t>(N0), static_cast<uint64_t>(N1)},
                          {N0 * e}, {kChunkK, static_cast<uint32_t>(p.N1p)});
  } else {
    tw1 = tw0;
  }
  p.out_box3 = map3(&to, D, static_cast<uint64_t>(M), Nout, kBlockM) ? 1 : 0;
  if (!p.out_box3)
    ok = ok && make_map(&to, D, p.is_bf16, 2,
                        {static_cast<uint64_t>(Nout), static_cast<uint64_t>(M)}, {Nout * e},
                        {64, kBlockM});
  if (!ok) return B2B_ERR_CUDA;
  p.pf_a = static_cast<const uint8_t*>(A);
  p.pf_a_bytes = static_cast<uint64_t>(M) * K0 * e;
  p.pf_a_tile_bytes = static_cast<uint32_t>(kBlockM * K0 * e);
  p.pf_w0 = static_cast<const uint8_t*>(W0);
  p.pf_w0_bytes = static_cast<uint32_t>(static_cast<uint64_t>(K0) * N0 * e);
  p.pf_w1 = static_cast<const uint8_t*>(W1);
  p.pf_w1_bytes = mode == MODE_CHAIN ? static_cast<uint32_t>(static_cast<uint64_t>(N0) * N1 * e) : 0u;
  p.out_ptr = static_cast<uint8_t*>(D);
  p.out_ld = Nout;
  Variant v;
  if (mode == MODE_CHAIN)
    v = !w_mn ? (p.p_tmem ? V_CONV1X1_CHAIN : V_CONV1X1_CHAIN_NP)
              : (p.p_split  ? V_GEMM_CHAIN_WIDE
                 : !p.p_tmem ? V_GEMM_CHAIN_NP
                 : p.w0_res  ? V_GEMM_CHAIN_PAIR_W0
                             : (!p.resident ? V_GEMM_CHAIN_PAIR : V_GEMM_CHAIN));
  else v = w_mn ? V_GEMM_SINGLE : V_CONV1X1_SINGLE;
  return launch(v, d, ta, tw0, tw1, to, p, smem, grid, stream);
}

// Three-operator chain (2-D A, row-major weights).
b2b_status run_gemm3_with(const Choice& ch, Info* info, int dt, int64_t M, int32_t K0, int32_t N0,
                          int32_t N1, int32_t N2, const void* A, const void* W0, const void* b0,
                          int e0, const void* W1, const void* b1, int e1, const void* W2,
                          const void* b2, int e2, void* D, void* stream) {
  ChainParams p;
  size_t smem = 0;
  Regions r;
  if (!gemm3_params(p, M, K0, N0, N1, N2, &smem, &r, ch.cand)) return B2B_ERR_UNSUPPORTED;
  b2b_status st = B2B_OK;
  DeviceState* d = device_state(&st);
  if (d == nullptr) return st;
  fill_common(p, dt, e0, e1, b0, b1, d, KID_GEMM_CHAIN3);
  p.act2 = e2;
  p.b2 = static_cast<const uint16_t*>(b2);
  p.w2 = static_cast<const uint16_t*>(W2);
  const int grid = grid_for(p.num_tiles, d->num_sms, ch.grid);
  p.pf_second = pf_second_for(p.num_tiles, grid, ch.pf2);
  if (info) *info = info_for(r, p.num_tiles, d->num_sms, true);

  CUtensorMap ta, tw0, tw1, to;
  const uint64_t e = 2;
  bool ok = make_map(&ta, A, p.is_bf16, 2, {static_cast<uint64_t>(K0), static_cast<uint64_t>(M)},
                     {K0 * e}, {kChunkK, kBlockM});
  // Row-major [rows][N] viewed as [N/64][rows][64] when N is a multiple of 64 (one box per
  // K chunk), else one 2-D box per 64-wide column block.
  auto wmap = [&](CUtensorMap* m, const void* ptr, uint64_t rows, int32_t N, uint32_t box_rows,
                  int32_t* box3) {
    *box3 = 0;
    if (N % 64 == 0 && make_map(m, ptr, p.is_bf16, 3, {64, rows, static_cast<uint64_t>(N / 64)},
                                {N * e, 128}, {64, box_rows, static_cast<uint32_t>(N / 64)})) {
      *box3 = 1;
      return true;
    }
    return make_map(m, ptr, p.is_bf16, 2, {static_cast<uint64_t>(N), rows}, {N * e},
                    {64, box_rows});
  };
  int32_t out3 = 0;
  ok = ok && wmap(&tw0, W0, static_cast<uint64_t>(K0), N0, 64, &p.w0_box3);
  ok = ok && wmap(&tw1, W1, static_cast<uint64_t>(N0), N1, 64, &p.w1_box3);
  ok = ok && wmap(&to, D, static_cast<uint64_t>(M), N2, kBlockM, &out3);
  p.out_box3 = out3;
  if (!ok) return B2B_ERR_CUDA;
  p.pf_a = static_cast<const uint8_t*>(A);
  p.pf_a_bytes = static_cast<uint64_t>(M) * K0 * e;
  p.pf_a_tile_bytes = static_cast<uint32_t>(kBlockM * K0 * e);
  p.pf_w0 = static_cast<const uint8_t*>(W0);
  p.pf_w0_bytes = static_cast<uint32_t>(static_cast<uint64_t>(K0) * N0 * e);
  p.pf_w1 = static_cast<const uint8_t*>(W1);
  p.pf_w1_bytes = static_cast<uint32_t>(static_cast<uint64_t>(N0) * N1 * e);
  return launch(V_GEMM_CHAIN3, d, ta, tw0, tw1, to, p, smem, grid, stream);
}

// ------------------------------------------------------------------------------------
// conv-shaped entry points (4-D implicit-GEMM A operand)
// ------------------------------------------------------------------------------------
// The conv + pool over CTA pairs (plan_pool_cta2): clusters of two CTAs, at most as many
// as can be resident at once; grid choices as for single CTAs, counted in pair-tiles.
b2b_status run_pool_cta2(const Choice& ch, Info* info, const Regions& r, ChainParams& p,
                         size_t smem, DeviceState* d, int32_t N, int32_t H, int32_t W, int32_t C,
                         const void* x, const void* W0, int32_t C0, int32_t R, int32_t S, void* y,
                         void* stream) {
  const bool traced = p.trace != nullptr;
  if (b2b_status st = ensure_smem_attribute(V_CONV_POOL_CTA2, d, p.is_bf16 != 0, traced);
      st != B2B_OK)
    return st;
  const int ci = 4 + (p.is_bf16 ? 1 : 0) + (traced ? 2 : 0);
  int clusters = d->cta2_clusters[ci].load();
  if (clusters <= 0 || d->cta2_smem[ci].load() != smem) {
    if (cta2_max_clusters(p.is_bf16 != 0, traced, smem, &clusters, true) != cudaSuccess ||
        clusters < 1) {
      cudaGetLastError();
      return B2B_ERR_CUDA;
    }
    d->cta2_clusters[ci].store(clusters);
    d->cta2_smem[ci].store(smem);
  }
  const int32_t pair_tiles = (p.num_tiles + 1) / 2;
  const int pairs = grid_for(pair_tiles, clusters, ch.grid);
  p.pf_second = 0;
  if (info) *info = info_for(r, pair_tiles, clusters, false);
  const uint64_t e = 2;
  CUtensorMap ta, tw0, to;
  // the halo box of each CTA's own tile, as the single-CTA kernel's
  bool ok = make_map(&ta, x, p.is_bf16, 4,
                     {static_cast<uint64_t>(C), static_cast<uint64_t>(W), static_cast<uint64_t>(H),
                      static_cast<uint64_t>(N)},
                     {C * e, static_cast<uint64_t>(W) * C * e, static_cast<uint64_t>(H) * W * C * e},
                     {kChunkK, 16, static_cast<uint32_t>(8 + R - 1), 1});
  // [C0][R*S][C]: half of the output channels (rows) of one tap's channel block per box
  ok = ok && make_map(&tw0, W0, p.is_bf16, 3,
                      {static_cast<uint64_t>(C), static_cast<uint64_t>(R) * S, static_cast<uint64_t>(C0)},
                      {C * e, static_cast<uint64_t>(R) * S * C * e},
                      {kChunkK, 1, static_cast<uint32_t>(p.N0p / 2)});
  const int32_t Hp = H / 2, Wp = W / 2;
  ok = ok && make_map(&to, y, p.is_bf16, 4,
                      {static_cast<uint64_t>(C0), static_cast<uint64_t>(Wp), static_cast<uint64_t>(Hp),
                       static_cast<uint64_t>(N)},
                      {C0 * e, static_cast<uint64_t>(Wp) * C0 * e, static_cast<uint64_t>(Hp) * Wp * C0 * e},
                      {64, 8, 4, 1});
  if (!ok) return B2B_ERR_CUDA;
  return launch(V_CONV_POOL_CTA2, d, ta, tw0, tw0, to, p, smem, 2 * pairs, stream);
}

b2b_status run_conv_with(const Choice& ch, Info* info, int mode, int dt, int32_t N, int32_t H,
                         int32_t W, int32_t C, const void* x, const void* W0, int32_t C0,
                         int32_t R, int32_t S, int32_t pad, int32_t stride, const void* b0, int e0,
                         const void* W1, int32_t C1, const void* b1, int e1, void* y,
                         void* stream, uint32_t kid) {
  ChainParams p;
  size_t smem = 0;
  Regions r;
  if (!conv_params(p, mode, N, H, W, C, C0, R, S, pad, C1, &smem, &r, ch.cand, stride))
    return B2B_ERR_UNSUPPORTED;
  b2b_status st = B2B_OK;
  DeviceState* d = device_state(&st);
  if (d == nullptr) return st;
  if (p.cta_pair) {
    fill_common(p, dt, e0, e1, b0, b1, d, KID_CONV_POOL_CTA2);
    return run_pool_cta2(ch, info, r, p, smem, d, N, H, W, C, x, W0, C0, R, S, y, stream);
  }
  fill_common(p, dt, e0, e1, b0, b1, d, kid);
  const int grid = grid_for(p.num_tiles, d->num_sms, ch.grid);
  p.pf_second = 0;   // the implicit-GEMM A has no per-tile contiguous range to prefetch
  if (r.extend > 0 && (p.num_tiles + grid - 1) / grid <= 2) p.num_stages += r.extend;
  if (info) *info = info_for(r, p.num_tiles, d->num_sms, false);
  const int32_t Ho = p.Ho, Wo = p.Wo;

  const uint64_t e = 2;
  CUtensorMap ta, tw0, tw1, to;
  // One box per (tap, channel block): 8 x 16 output pixels, i.e. input pixels `stride`
  // apart (the box spans 8 * stride x 16 * stride pixels and takes every stride-th); halo
  // boxes (stride 1, resident filters) take 8 + R - 1 rows for all row taps.
  const uint32_t sd = static_cast<uint32_t>(stride);
  bool ok = make_map(&ta, x, p.is_bf16, 4,
                     {static_cast<uint64_t>(C), static_cast<uint64_t>(W), static_cast<uint64_t>(H),
                      static_cast<uint64_t>(N)},
                     {C * e, static_cast<uint64_t>(W) * C * e, static_cast<uint64_t>(H) * W * C * e},
                     {kChunkK, 16 * sd, static_cast<uint32_t>(p.halo ? 8 + R - 1 : 8 * sd), 1},
                     {1, sd, sd, 1});
  ok = ok && make_map(&tw0, W0, p.is_bf16, 3,
                      {static_cast<uint64_t>(C), static_cast<uint64_t>(R) * S, static_cast<uint64_t>(C0)},
                      {C * e, static_cast<uint64_t>(R) * S * C * e},
                      {kChunkK, 1, static_cast<uint32_t>(p.N0p)});
  if (mode == MODE_CHAIN)
    ok = ok && make_map(&tw1, W1, p.is_bf16, 2, {static_cast<uint64_t>(C0), static_cast<uint64_t>(C1)},
                        {C0 * e}, {kChunkK, static_cast<uint32_t>(p.N1p)});
  else
    tw1 = tw0;
  if (mode == MODE_POOL) {
    const int32_t Hp = H / 2, Wp = W / 2;
    ok = ok && make_map(&to, y, p.is_bf16, 4,
                        {static_cast<uint64_t>(C0), static_cast<uint64_t>(Wp), static_cast<uint64_t>(Hp),
                         static_cast<uint64_t>(N)},
                        {C0 * e, static_cast<uint64_t>(Wp) * C0 * e, static_cast<uint64_t>(Hp) * Wp * C0 * e},
                        {64, 8, 4, 1});
  } else {
    const int32_t Cout = mode == MODE_CHAIN ? C1 : C0;
    ok = ok && make_map(&to, y, p.is_bf16, 4,
                        {static_cast<uint64_t>(Cout), static_cast<uint64_t>(Wo), static_cast<uint64_t>(Ho),
                         static_cast<uint64_t>(N)},
                        {Cout * e, static_cast<uint64_t>(Wo) * Cout * e, static_cast<uint64_t>(Ho) * Wo * Cout * e},
                        {64, 16, 8, 1});
  }
  if (!ok) return B2B_ERR_CUDA;
  p.pf_w0 = static_cast<const uint8_t*>(W0);
  p.pf_w0_bytes = static_cast<uint32_t>(static_cast<uint64_t>(C0) * R * S * C * e);
  p.pf_w1 = static_cast<const uint8_t*>(W1);
  p.pf_w1_bytes = mode == MODE_CHAIN ? static_cast<uint32_t>(static_cast<uint64_t>(C1) * C0 * e) : 0u;
  // The two-issuer chain stores each warp's 32 rows (two output rows of 16 pixels) 16
  // channels at a time from its own 1 KiB slot.
  if (p.out_slots)
    ok = ok && make_map(&to, y, p.is_bf16, 4,
                        {static_cast<uint64_t>(C1), static_cast<uint64_t>(Wo), static_cast<uint64_t>(Ho),
                         static_cast<uint64_t>(N)},
                        {C1 * e, static_cast<uint64_t>(Wo) * C1 * e, static_cast<uint64_t>(Ho) * Wo * C1 * e},
                        {16, 16, 2, 1}, {1, 1, 1, 1}, false);
  if (!ok) return B2B_ERR_CUDA;
  const Variant v = mode == MODE_CHAIN    ? (p.two_issuers ? V_CONV_CHAIN_2I
                                            : p.p_tmem    ? V_CONV_CHAIN
                                                          : V_CONV_CHAIN_NP)
                    : mode == MODE_SINGLE ? V_CONV_SINGLE
                                          : V_CONV_POOL;
  return launch(v, d, ta, tw0, tw1, to, p, smem, grid, stream);
}

// ------------------------------------------------------------------------------------
// light-weight profiler (BOLT notes, "Light-weight performance profiler": a search over
// launch parameters by timing): per problem, time every launch choice once, keep the fastest
// ------------------------------------------------------------------------------------
// Problems are keyed by the entry point, its sizes (as b2b_debug_plan takes them) and,
// last, its variant: the dtype and epilogue kinds, which select different kernel
// instantiations (kAnyVariant: a choice pinned or ranked for every variant of the sizes).
using TuneKey = std::vector<int64_t>;
constexpr int64_t kAnyVariant = -1;

int64_t variant_of(int dt, int e0 = 0, int e1 = 0, int e2 = 0) {
  return static_cast<int64_t>(dt) | (static_cast<int64_t>(e0) << 4) |
         (static_cast<int64_t>(e1) << 8) | (static_cast<int64_t>(e2) << 12);
}

TuneKey any_variant(TuneKey k) {
  k.back() = kAnyVariant;
  return k;
}

// One timed launch choice: the layout, grid mode and the CTAs it gave, the second-tile
// prefetch (-1: the default rule) and the fastest round's time per launch.
struct TimedChoice {
  int32_t cand, grid, ctas, pf2, ns;
};

struct Tuned {
  Choice c;
  int32_t source = 0;   // 1 pinned by b2b_set_choice, 2 measured, 3 ranked by b2b_set_candidates
  uint32_t best_ns = 0, default_ns = 0, timed = 0;
  uint64_t seq = 0;                  // order of recording (the most recent wins a wildcard query)
  std::vector<int32_t> cands;        // source 3: the layouts to time, the first the default
  std::vector<TimedChoice> record;   // source 2: every choice timed, the default first
};

std::mutex g_tune_mu;
std::map<TuneKey, Tuned> g_tuned;
uint64_t g_tune_seq = 0;
std::atomic<int> g_autotune{0};
// Per choice: kTuneWarm untimed launches, then kTuneRounds rounds of kTuneReps launches;
// a choice's time is its fastest round.  Another choice replaces the default only when
// it is faster by more than kTuneMargin (timing noise must not pick a layout).
constexpr int kTuneWarm = 2, kTuneReps = 10, kTuneRounds = 3;
constexpr float kTuneMargin = 0.02f;

// The entry recorded for a call's key: its own variant's, else one for every variant.
bool find_tuned(const TuneKey& key, Tuned* t) {
  std::lock_guard<std::mutex> lk(g_tune_mu);
  auto it = g_tuned.find(key);
  if (it == g_tuned.end() && key.back() != kAnyVariant) it = g_tuned.find(any_variant(key));
  if (it == g_tuned.end()) return false;
  *t = it->second;
  return true;
}

// A query for a variant: its own entry, else the one for every variant of its sizes (what
// its calls take).  A query by sizes alone (kAnyVariant): the most recently recorded entry
// of those sizes, for every variant or for one.  Caller holds g_tune_mu.
const Tuned* find_for_query(const TuneKey& key) {
  if (key.back() != kAnyVariant) {
    auto it = g_tuned.find(key);
    if (it == g_tuned.end()) it = g_tuned.find(any_variant(key));
    return it == g_tuned.end() ? nullptr : &it->second;
  }
  const Tuned* best = nullptr;
  for (auto j = g_tuned.lower_bound(key); j != g_tuned.end(); ++j) {
    if (!std::equal(key.begin(), key.end() - 1, j->first.begin(), j->first.end() - 1)) break;
    if (best == nullptr || j->second.seq > best->seq) best = &j->second;
  }
  return best;
}

bool find_choice(const TuneKey& key, Choice* c) {
  std::lock_guard<std::mutex> lk(g_tune_mu);
  const Tuned* t = find_for_query(key);
  if (t == nullptr) return false;
  *c = t->c;
  return true;
}

// Times `go(choice)` for the default and for every layout x grid x prefetch choice that
// differs from it in effect, on the caller's stream (which it synchronises), records the
// fastest (and every time) under `key` and launches it for the caller.  `cands`, if not
// empty, restricts the layouts to those (a model's ranking) and makes the first the default.
template <class Go>
b2b_status tune(const TuneKey& key, void* stream, Go&& go, const std::vector<int32_t>& cands) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Choice def = cands.empty() ? Choice{} : Choice{cands[0], -1, -1};
  Info info;
  b2b_status st = go(def, &info);
  if (st != B2B_OK) return st;
  cudaEvent_t ev0 = nullptr, ev1 = nullptr;
  if (cudaEventCreate(&ev0) != cudaSuccess || cudaEventCreate(&ev1) != cudaSuccess) {
    cudaGetLastError();
    if (ev0) cudaEventDestroy(ev0);
    return B2B_ERR_CUDA;
  }
  auto time_of = [&](const Choice& c, float* us) -> b2b_status {
    for (int i = 0; i < kTuneWarm; ++i)
      if (b2b_status e = go(c, nullptr); e != B2B_OK) return e;
    for (int round = 0; round < kTuneRounds; ++round) {
      if (cudaEventRecord(ev0, s) != cudaSuccess) return B2B_ERR_CUDA;
      for (int i = 0; i < kTuneReps; ++i)
        if (b2b_status e = go(c, nullptr); e != B2B_OK) return e;
      float ms = 0.f;
      if (cudaEventRecord(ev1, s) != cudaSuccess || cudaEventSynchronize(ev1) != cudaSuccess ||
          cudaEventElapsedTime(&ms, ev0, ev1) != cudaSuccess)
        return B2B_ERR_CUDA;
      const float t = ms * 1000.f / kTuneReps;
      if (round == 0 || t < *us) *us = t;
    }
    return B2B_OK;
  };
  std::vector<int32_t> layouts = cands;
  if (layouts.empty())
    for (int32_t c = 0; c < info.ncand; ++c) layouts.push_back(c);
  float def_us = 0.f, best_us = 0.f;
  Choice best = def;
  std::vector<TimedChoice> record;
  st = time_of(def, &def_us);
  if (st == B2B_OK) {
    best_us = def_us;
    record.push_back({info.cand, 0, info.grid[0], -1, static_cast<int32_t>(def_us * 1000.f)});
    for (size_t li = 0; li < layouts.size() && st == B2B_OK; ++li)
      for (int32_t grid = 0; grid < kGridModes && st == B2B_OK; ++grid) {
        const int32_t cand = layouts[li];
        bool same = false;   // a grid mode that gives an earlier mode's grid is skipped
        for (int m = 0; m < grid; ++m) same = same || info.grid[m] == info.grid[grid];
        if (same) continue;
        // the second-tile prefetch matters only where some CTA has a second tile
        const int pfs = (info.can_prefetch && info.tiles > info.grid[grid]) ? 2 : 1;
        for (int32_t pf = 0; pf < pfs && st == B2B_OK; ++pf) {
          const Choice c{cand, grid, pfs == 2 ? pf : 0};
          float us = 0.f;
          st = time_of(c, &us);
          if (st == B2B_OK) {
            record.push_back({cand, grid, info.grid[grid], c.pf2, static_cast<int32_t>(us * 1000.f)});
            if (us < best_us && us < def_us * (1.f - kTuneMargin)) {
              best = c;
              best_us = us;
            }
          }
        }
      }
  }
  if (st == B2B_ERR_CUDA) cudaGetLastError();
  cudaEventDestroy(ev0);
  cudaEventDestroy(ev1);
  if (st != B2B_OK) return st;
  {
    std::lock_guard<std::mutex> lk(g_tune_mu);
    Tuned& t = g_tuned[key];
    t = Tuned{};
    t.c = best;
    t.source = 2;
    t.best_ns = static_cast<uint32_t>(best_us * 1000.f);
    t.default_ns = static_cast<uint32_t>(def_us * 1000.f);
    t.timed = static_cast<uint32_t>(record.size());
    t.seq = ++g_tune_seq;
    t.cands = cands;
    t.record = std::move(record);
  }
  return go(best, nullptr);
}

// The launch choice of a problem: pinned or measured before, else (with the profiler on,
// outside stream capture) measured now over the top layouts of a ranking -- the caller's
// (b2b_set_candidates) or the tile-graph model's -- else that ranking's first layout.
template <class Go>
b2b_status dispatch(const TuneKey& key, void* stream, Go&& go) {
  Tuned t;
  const bool have = find_tuned(key, &t);
  if (have && t.source != 3) {
    if (t.c.cand < 0) {   // a pinned grid or prefetch alone: the model's layout
      std::vector<int32_t> top;
      if (b2b_status st = model_top(key, &top); st != B2B_OK) return st;
      t.c.cand = top[0];
    }
    return go(t.c, nullptr);
  }
  std::vector<int32_t> cands;
  if (have) {
    cands = t.cands;
  } else if (b2b_status st = model_top(key, &cands); st != B2B_OK) {
    return st;
  }
  const Choice c{cands[0], -1, -1};
  if (g_autotune.load() == 0) return go(c, nullptr);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cs) != cudaSuccess) {
    cudaGetLastError();
    return B2B_ERR_CUDA;
  }
  if (cs != cudaStreamCaptureStatusNone) return go(c, nullptr);
  return tune(key, stream, go, cands);
}

b2b_status run_gemm(const TuneKey& key, int mode, bool w_mn, int dt, int64_t M, int32_t K0,
                    int32_t N0, int32_t N1, const void* A, const void* W0, const void* b0, int e0,
                    const void* W1, const void* b1, int e1, void* D, void* stream, uint32_t kid) {
  return dispatch(key, stream, [&](const Choice& c, Info* info) {
    return run_gemm_with(c, info, mode, w_mn, dt, M, K0, N0, N1, A, W0, b0, e0, W1, b1, e1, D,
                         stream, kid);
  });
}

b2b_status run_gemm3(const TuneKey& key, int dt, int64_t M, int32_t K0, int32_t N0, int32_t N1,
                     int32_t N2, const void* A, const void* W0, const void* b0, int e0,
                     const void* W1, const void* b1, int e1, const void* W2, const void* b2,
                     int e2, void* D, void* stream) {
  return dispatch(key, stream, [&](const Choice& c, Info* info) {
    return run_gemm3_with(c, info, dt, M, K0, N0, N1, N2, A, W0, b0, e0, W1, b1, e1, W2, b2, e2,
                          D, stream);
  });
}

b2b_status run_conv(const TuneKey& key, int mode, int dt, int32_t N, int32_t H, int32_t W,
                    int32_t C, const void* x, const void* W0, int32_t C0, int32_t R, int32_t S,
                    int32_t pad, int32_t stride, const void* b0, int e0, const void* W1,
                    int32_t C1, const void* b1, int e1, void* y, void* stream, uint32_t kid) {
  return dispatch(key, stream, [&](const Choice& c, Info* info) {
    return run_conv_with(c, info, mode, dt, N, H, W, C, x, W0, C0, R, S, pad, stride, b0, e0, W1,
                         C1, b1, e1, y, stream, kid);
  });
}

// Shared checks of a channel-like size: multiple of 8 (16 bytes), within [8, hi].
b2b_status check_channels(int32_t c, int32_t hi) {
  if (c < 8) return c <= 0 ? B2B_ERR_SHAPE : B2B_ERR_ALIGN;
  if (c % 8 != 0) return B2B_ERR_ALIGN;
  if (c > hi) return B2B_ERR_UNSUPPORTED;
  return B2B_OK;
}

constexpr int32_t kMaxReduction = 1 << 16;   // K0 or C: keeps all index math in int32

}  // namespace
}  // namespace b2b

using namespace b2b;

extern "C" {

b2b_status b2b_gemm(b2b_dtype dt, int64_t M, int32_t K0, int32_t N0, int32_t N1, const void* A,
                    const void* W0, const void* b0, b2b_epilogue e0, const void* W1,
                    const void* b1, b2b_epilogue e1, void* D, void* stream) {
  if (!valid_dtype(dt) || !valid_epi(e0) || !valid_epi(e1)) return B2B_ERR_UNSUPPORTED;
  if (M < 0 || K0 <= 0 || N0 <= 0 || N1 <= 0) return B2B_ERR_SHAPE;
  b2b_status st;
  if ((st = check_channels(K0, kMaxReduction)) != B2B_OK) return st;
  if ((st = check_channels(N0, 512)) != B2B_OK) return st;
  if ((st = check_channels(N1, 256)) != B2B_OK) return st;
  if (M > static_cast<int64_t>(INT32_MAX) - kBlockM) return B2B_ERR_UNSUPPORTED;
  if (M == 0) return B2B_OK;
  if (!A || !W0 || !W1 || !D) return B2B_ERR_NULL;
  if (!aligned16(A) || !aligned16(W0) || !aligned16(W1) || !aligned16(D)) return B2B_ERR_ALIGN;
  if ((b0 && !aligned2(b0)) || (b1 && !aligned2(b1))) return B2B_ERR_ALIGN;
  return run_gemm({0, M, K0, N0, N1, variant_of(dt, e0, e1)}, MODE_CHAIN, true, dt, M, K0, N0, N1, A, W0, b0, e0, W1, b1,
                  e1, D, stream, KID_GEMM_CHAIN);
}

b2b_status b2b_gemm3(b2b_dtype dt, int64_t M, int32_t K0, int32_t N0, int32_t N1, int32_t N2,
                     const void* A, const void* W0, const void* b0, b2b_epilogue e0,
                     const void* W1, const void* b1, b2b_epilogue e1, const void* W2,
                     const void* b2, b2b_epilogue e2, void* D, void* stream) {
  if (!valid_dtype(dt) || !valid_epi(e0) || !valid_epi(e1) || !valid_epi(e2))
    return B2B_ERR_UNSUPPORTED;
  if (M < 0 || K0 <= 0 || N0 <= 0 || N1 <= 0 || N2 <= 0) return B2B_ERR_SHAPE;
  b2b_status st;
  if ((st = check_channels(K0, kMaxReduction)) != B2B_OK) return st;
  if ((st = check_channels(N0, 256)) != B2B_OK) return st;
  if ((st = check_channels(N1, 256)) != B2B_OK) return st;
  if ((st = check_channels(N2, 256)) != B2B_OK) return st;
  if (M > static_cast<int64_t>(INT32_MAX) - kBlockM) return B2B_ERR_UNSUPPORTED;
  if (M == 0) return B2B_OK;
  if (!A || !W0 || !W1 || !W2 || !D) return B2B_ERR_NULL;
  if (!aligned16(A) || !aligned16(W0) || !aligned16(W1) || !aligned16(W2) || !aligned16(D))
    return B2B_ERR_ALIGN;
  if ((b0 && !aligned2(b0)) || (b1 && !aligned2(b1)) || (b2 && !aligned2(b2)))
    return B2B_ERR_ALIGN;
  return run_gemm3({5, M, K0, N0, N1, N2, variant_of(dt, e0, e1, e2)}, dt, M, K0, N0, N1, N2, A, W0, b0, e0, W1, b1, e1, W2,
                   b2, e2, D, stream);
}

b2b_status gemm_bias_act(b2b_dtype dt, int64_t M, int32_t K, int32_t N, const void* A,
                         const void* W, const void* b, b2b_epilogue e, void* D, void* stream) {
  if (!valid_dtype(dt) || !valid_epi(e)) return B2B_ERR_UNSUPPORTED;
  if (M < 0 || K <= 0 || N <= 0) return B2B_ERR_SHAPE;
  b2b_status st;
  if ((st = check_channels(K, kMaxReduction)) != B2B_OK) return st;
  if ((st = check_channels(N, 256)) != B2B_OK) return st;
  if (M > static_cast<int64_t>(INT32_MAX) - kBlockM) return B2B_ERR_UNSUPPORTED;
  if (M == 0) return B2B_OK;
  if (!A || !W || !D) return B2B_ERR_NULL;
  if (!aligned16(A) || !aligned16(W) || !aligned16(D)) return B2B_ERR_ALIGN;
  if (b && !aligned2(b)) return B2B_ERR_ALIGN;
  return run_gemm({1, M, K, N, variant_of(dt, e)}, MODE_SINGLE, true, dt, M, K, N, 0, A, W, b, e, nullptr, nullptr, 0,
                  D, stream, KID_GEMM_SINGLE);
}

static b2b_status check_conv_args(int32_t N, int32_t H, int32_t W, int32_t C, int32_t Co,
                                  int32_t R, int32_t S, int32_t pad, int32_t stride = 1) {
  if (N < 0 || H < 0 || W < 0) return B2B_ERR_SHAPE;
  b2b_status st;
  if ((st = check_channels(C, kMaxReduction)) != B2B_OK) return st;
  if ((st = check_channels(Co, 256)) != B2B_OK) return st;
  if (R < 1 || S < 1 || pad < 0 || stride < 1) return B2B_ERR_SHAPE;
  if (R > 7 || S > 7 || pad > 3 || stride > 4) return B2B_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(R) * S * ((C + 63) / 64) > 4096) return B2B_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(N) * H * W > 0) {
    if (H + 2 * pad - R + 1 < 1 || W + 2 * pad - S + 1 < 1) return B2B_ERR_SHAPE;
  }
  if (static_cast<int64_t>(N) * H * W * C > (int64_t{1} << 40)) return B2B_ERR_UNSUPPORTED;
  return B2B_OK;
}

b2b_status b2b_conv_nhwc_strided(b2b_dtype dt, int32_t N, int32_t H, int32_t W, int32_t C,
                                 const void* x, const void* W0, int32_t C0, int32_t R, int32_t S,
                                 int32_t pad, int32_t stride, const void* b0, b2b_epilogue e0,
                                 const void* W1, int32_t C1, const void* b1, b2b_epilogue e1,
                                 void* y, void* stream) {
  if (!valid_dtype(dt) || !valid_epi(e0) || !valid_epi(e1)) return B2B_ERR_UNSUPPORTED;
  b2b_status st = check_conv_args(N, H, W, C, C0, R, S, pad, stride);
  if (st != B2B_OK) return st;
  if ((st = check_channels(C1, 256)) != B2B_OK) return st;
  if (static_cast<int64_t>(N) * H * W == 0) return B2B_OK;
  if (!x || !W0 || !W1 || !y) return B2B_ERR_NULL;
  if (!aligned16(x) || !aligned16(W0) || !aligned16(W1) || !aligned16(y)) return B2B_ERR_ALIGN;
  if ((b0 && !aligned2(b0)) || (b1 && !aligned2(b1))) return B2B_ERR_ALIGN;
  const TuneKey key{2, N, H, W, C, C0, R, S, pad, C1, stride, variant_of(dt, e0, e1)};
  if (R == 1 && S == 1 && pad == 0 && stride == 1) {
    // A 1x1 conv is a GEMM over the N*H*W pixel rows (interview notes, "Conv
    // optimisation", item 5): run the GEMM-shaped kernel with K-major filters.
    const int64_t M = static_cast<int64_t>(N) * H * W;
    if (M > static_cast<int64_t>(INT32_MAX) - kBlockM) return B2B_ERR_UNSUPPORTED;
    return run_gemm(key, MODE_CHAIN, false, dt, M, C, C0, C1, x, W0, b0, e0, W1, b1, e1, y, stream,
                    KID_CONV1X1_CHAIN);
  }
  return run_conv(key, MODE_CHAIN, dt, N, H, W, C, x, W0, C0, R, S, pad, stride, b0, e0, W1, C1, b1,
                  e1, y, stream, KID_CONV_CHAIN);
}

b2b_status b2b_conv_nhwc(b2b_dtype dt, int32_t N, int32_t H, int32_t W, int32_t C, const void* x,
                         const void* W0, int32_t C0, int32_t R, int32_t S, int32_t pad,
                         const void* b0, b2b_epilogue e0, const void* W1, int32_t C1,
                         const void* b1, b2b_epilogue e1, void* y, void* stream) {
  return b2b_conv_nhwc_strided(dt, N, H, W, C, x, W0, C0, R, S, pad, 1, b0, e0, W1, C1, b1, e1, y,
                               stream);
}

b2b_status conv_bias_act_nhwc_strided(b2b_dtype dt, int32_t N, int32_t H, int32_t W, int32_t C,
                                      const void* x, const void* Wt, int32_t Co, int32_t R,
                                      int32_t S, int32_t pad, int32_t stride, const void* b,
                                      b2b_epilogue e, void* y, void* stream) {
  if (!valid_dtype(dt) || !valid_epi(e)) return B2B_ERR_UNSUPPORTED;
  b2b_status st = check_conv_args(N, H, W, C, Co, R, S, pad, stride);
  if (st != B2B_OK) return st;
  if (static_cast<int64_t>(N) * H * W == 0) return B2B_OK;
  if (!x || !Wt || !y) return B2B_ERR_NULL;
  if (!aligned16(x) || !aligned16(Wt) || !aligned16(y)) return B2B_ERR_ALIGN;
  if (b && !aligned2(b)) return B2B_ERR_ALIGN;
  const TuneKey key{3, N, H, W, C, Co, R, S, pad, stride, variant_of(dt, e)};
  if (R == 1 && S == 1 && pad == 0 && stride == 1) {
    const int64_t M = static_cast<int64_t>(N) * H * W;
    if (M > static_cast<int64_t>(INT32_MAX) - kBlockM) return B2B_ERR_UNSUPPORTED;
    return run_gemm(key, MODE_SINGLE, false, dt, M, C, Co, 0, x, Wt, b, e, nullptr, nullptr, 0, y,
                    stream, KID_CONV1X1_SINGLE);
  }
  return run_conv(key, MODE_SINGLE, dt, N, H, W, C, x, Wt, Co, R, S, pad, stride, b, e, nullptr, 0,
                  nullptr, 0, y, stream, KID_CONV_SINGLE);
}

b2b_status conv_bias_act_nhwc(b2b_dtype dt, int32_t N, int32_t H, int32_t W, int32_t C,
                              const void* x, const void* Wt, int32_t Co, int32_t R, int32_t S,
                              int32_t pad, const void* b, b2b_epilogue e, void* y, void* stream) {
  return conv_bias_act_nhwc_strided(dt, N, H, W, C, x, Wt, Co, R, S, pad, 1, b, e, y, stream);
}

b2b_status conv_relu_maxpool(b2b_dtype dt, int32_t N, int32_t H, int32_t W, int32_t Cin,
                             const void* x, const void* Wt, const void* b, int32_t Cout, void* y,
                             void* stream) {
  if (!valid_dtype(dt)) return B2B_ERR_UNSUPPORTED;
  if (N < 0 || H < 0 || W < 0) return B2B_ERR_SHAPE;
  if (N > 0 && (H < 2 || W < 2)) return B2B_ERR_SHAPE;
  b2b_status st = check_conv_args(N, H, W, Cin, Cout, 3, 3, 1);
  if (st != B2B_OK) return st;
  if (N == 0) return B2B_OK;
  if (!x || !Wt || !y) return B2B_ERR_NULL;
  if (!aligned16(x) || !aligned16(Wt) || !aligned16(y)) return B2B_ERR_ALIGN;
  if (b && !aligned2(b)) return B2B_ERR_ALIGN;
  return run_conv({4, N, H, W, Cin, Cout, variant_of(dt)}, MODE_POOL, dt, N, H, W, Cin, x, Wt, Cout, 3, 3, 1, 1, b,
                  B2B_EPI_RELU, nullptr, 0, nullptr, 0, y, stream, KID_CONV_POOL);
}

b2b_status b2b_fold_batchnorm(b2b_dtype dt, int64_t Co, int64_t K, int32_t out_inner,
                              const void* Wt, const void* b, const float* gamma,
                              const float* beta, const float* mean, const float* var, float eps,
                              void* W_out, void* b_out, void* stream) {
  if (!valid_dtype(dt) || (out_inner != 0 && out_inner != 1)) return B2B_ERR_UNSUPPORTED;
  if (Co <= 0 || K <= 0 || !(eps >= 0.f) || Co > (int64_t{1} << 40) / K) return B2B_ERR_SHAPE;
  if (!Wt || !gamma || !beta || !mean || !var || !W_out || !b_out) return B2B_ERR_NULL;
  auto al = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
  if (!al(Wt, 2) || !al(W_out, 2) || !al(b_out, 2) || (b && !al(b, 2)) || !al(gamma, 4) ||
      !al(beta, 4) || !al(mean, 4) || !al(var, 4))
    return B2B_ERR_ALIGN;
  b2b_status st = B2B_OK;
  DeviceState* d = device_state(&st);
  if (d == nullptr) return st;
  if (launch_fold_batchnorm(dt == B2B_BF16, Co, K, out_inner, Wt, b, gamma, beta, mean, var, eps,
                            W_out, b_out, d->num_sms, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess) {
    cudaGetLastError();
    return B2B_ERR_CUDA;
  }
  return B2B_OK;
}

b2b_status maxpool2x2_nhwc(b2b_dtype dt, int32_t N, int32_t H, int32_t W, int32_t C,
                           const void* x, void* y, void* stream) {
  if (!valid_dtype(dt)) return B2B_ERR_UNSUPPORTED;
  if (N < 0 || H < 0 || W < 0 || C <= 0) return B2B_ERR_SHAPE;
  if (N > 0 && (H < 2 || W < 2)) return B2B_ERR_SHAPE;
  if (C % 8 != 0) return B2B_ERR_ALIGN;
  if (N == 0) return B2B_OK;
  if (!x || !y) return B2B_ERR_NULL;
  if (!aligned16(x) || !aligned16(y)) return B2B_ERR_ALIGN;
  b2b_status st = B2B_OK;
  DeviceState* d = device_state(&st);
  if (d == nullptr) return st;
  if (launch_maxpool(dt == B2B_BF16, N, H, W, C, x, y, d->num_sms,
                     static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return B2B_ERR_CUDA;
  }
  return B2B_OK;
}

const char* b2b_status_str(b2b_status s) {
  switch (s) {
    case B2B_OK: return "B2B_OK";
    case B2B_ERR_NULL: return "B2B_ERR_NULL: a required pointer is NULL";
    case B2B_ERR_SHAPE: return "B2B_ERR_SHAPE: invalid or inconsistent size";
    case B2B_ERR_ALIGN: return "B2B_ERR_ALIGN: pointer not 16-byte aligned or size not a multiple of 8";
    case B2B_ERR_UNSUPPORTED: return "B2B_ERR_UNSUPPORTED: outside the kernels' limits";
    case B2B_ERR_CUDA: return "B2B_ERR_CUDA: a CUDA call failed";
    case B2B_ERR_TIMEOUT: return "B2B_ERR_TIMEOUT: a kernel gave up waiting";
    default: return "unknown b2b_status";
  }
}

const char* b2b_version(void) { return "0.1.0"; }

int32_t b2b_num_sms(void) {
  b2b_status st = B2B_OK;
  DeviceState* d = device_state(&st);
  return d ? d->num_sms : -1;
}

void b2b_set_wait_limit_ns(uint64_t ns) { g_wait_ns.store(ns == 0 ? kDefaultWaitNs : ns); }

b2b_status b2b_set_trace(void* buf, uint32_t capacity, uint32_t cta) {
  if (buf != nullptr && (reinterpret_cast<uintptr_t>(buf) & 7u) != 0) return B2B_ERR_ALIGN;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_buf = static_cast<unsigned long long*>(buf);
  g_trace_cap = buf ? capacity : 0u;
  g_trace_cta = cta;
  return B2B_OK;
}

b2b_status b2b_get_device_error(uint32_t info[4]) {
  b2b_status st = B2B_OK;
  DeviceState* d = device_state(&st);
  if (d == nullptr) return st;
  uint32_t w[4] = {0, 0, 0, 0};
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(w, d->err, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return B2B_ERR_CUDA;
  }
  if (info) std::memcpy(info, w, sizeof(w));
  if (w[0] == 0u) return B2B_OK;
  const uint32_t zero[4] = {0, 0, 0, 0};
  if (cudaMemcpy(d->err, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return B2B_ERR_CUDA;
  }
  return w[0] == ERR_CODE_TIMEOUT ? B2B_ERR_TIMEOUT : B2B_ERR_CUDA;
}

// Sizes an entry point takes, per kind (b2b_debug_plan's numbering), and its epilogue kinds.
static const int32_t kPlanDims[6] = {4, 3, 9, 8, 5, 5};
static const int32_t kPlanActs[6] = {2, 1, 2, 1, 0, 3};

static bool plan_is_conv(int32_t kind) { return kind == 2 || kind == 3; }

// Where the optional variant (dtype, then each epilogue kind) starts in dims: after the
// sizes and, for the convs, the stride (which must then be given).
static int32_t plan_variant_at(int32_t kind) { return kPlanDims[kind] + (plan_is_conv(kind) ? 1 : 0); }

// The convs (kinds 2 and 3) take an optional stride after their sizes (default 1).
static int64_t plan_stride(int32_t kind, const int64_t* dims, int32_t ndims) {
  return (plan_is_conv(kind) && ndims > kPlanDims[kind]) ? dims[kPlanDims[kind]] : 1;
}

static bool plan_has_variant(int32_t kind, int32_t ndims) { return ndims > plan_variant_at(kind); }

static b2b_status check_plan_args(int32_t kind, const int64_t* dims, int32_t ndims) {
  if (kind < 0 || kind > 5) return B2B_ERR_UNSUPPORTED;
  if (dims == nullptr) return B2B_ERR_NULL;
  const int32_t base = kPlanDims[kind], at = plan_variant_at(kind);
  if (ndims < base) return B2B_ERR_SHAPE;
  if (ndims > at && ndims != at + 1 + kPlanActs[kind]) return B2B_ERR_SHAPE;
  for (int i = 0; i < base; ++i)
    if (dims[i] < 0 || dims[i] > INT32_MAX) return B2B_ERR_SHAPE;
  const int64_t st = plan_stride(kind, dims, ndims);
  if (st < 1 || st > INT32_MAX) return B2B_ERR_SHAPE;
  if (plan_has_variant(kind, ndims)) {
    if (dims[at] < 0 || dims[at] > 1 || !valid_dtype(static_cast<int>(dims[at])))
      return B2B_ERR_SHAPE;
    for (int a = 0; a < kPlanActs[kind]; ++a)
      if (dims[at + 1 + a] < 0 || dims[at + 1 + a] > 2) return B2B_ERR_SHAPE;
  }
  return B2B_OK;
}

// The key the entry point files its launch choice under (the convs' with their stride),
// for the variant dims names, else for every variant.
static TuneKey plan_key(int32_t kind, const int64_t* dims, int32_t ndims) {
  TuneKey k{kind};
  k.insert(k.end(), dims, dims + kPlanDims[kind]);
  if (plan_is_conv(kind)) k.push_back(plan_stride(kind, dims, ndims));
  if (!plan_has_variant(kind, ndims)) {
    k.push_back(kAnyVariant);
    return k;
  }
  const int32_t at = plan_variant_at(kind);
  int e[3] = {0, 0, 0};
  // conv_relu_maxpool's epilogue is fixed (ReLU), as its entry point files it
  for (int a = 0; a < kPlanActs[kind]; ++a) e[a] = static_cast<int>(dims[at + 1 + a]);
  k.push_back(variant_of(static_cast<int>(dims[at]), e[0], e[1], e[2]));
  return k;
}

// The launch plan entry point `kind` makes for `dims` with layout candidate `forced`
// (-1: the planner's default); validated like the entry point itself.
static b2b_status plan_for_kind(int32_t kind, const int64_t* dims, int32_t ndims, int forced,
                                ChainParams& p, Regions& r, size_t& smem, int32_t& mode) {
  const int32_t d0 = static_cast<int32_t>(dims[0]), d1 = static_cast<int32_t>(dims[1]),
                d2 = static_cast<int32_t>(dims[2]), d3 = static_cast<int32_t>(dims[3]);
  bool ok = false;
  b2b_status st = B2B_OK;
  mode = MODE_CHAIN;
  switch (kind) {
    case 0:   // b2b_gemm: M, K0, N0, N1
      if ((st = check_channels(d1, kMaxReduction)) != B2B_OK) return st;
      if ((st = check_channels(d2, 512)) != B2B_OK) return st;
      if ((st = check_channels(d3, 256)) != B2B_OK) return st;
      ok = gemm_params(p, MODE_CHAIN, true, dims[0], d1, d2, d3, &smem, &r, forced);
      break;
    case 1:   // gemm_bias_act: M, K, N
      if ((st = check_channels(d1, kMaxReduction)) != B2B_OK) return st;
      if ((st = check_channels(d2, 256)) != B2B_OK) return st;
      mode = MODE_SINGLE;
      ok = gemm_params(p, MODE_SINGLE, true, dims[0], d1, d2, 0, &smem, &r, forced);
      break;
    case 2:
    case 3: {  // b2b_conv_nhwc: N,H,W,C,C0,R,S,pad[,C1]; conv_bias_act_nhwc: N,H,W,C,Co,R,S,pad
      const int32_t C0 = static_cast<int32_t>(dims[4]), R = static_cast<int32_t>(dims[5]),
                    S = static_cast<int32_t>(dims[6]), pad = static_cast<int32_t>(dims[7]);
      const int32_t C1 = kind == 2 ? static_cast<int32_t>(dims[8]) : 0;
      const int32_t stride = static_cast<int32_t>(plan_stride(kind, dims, ndims));
      if ((st = check_conv_args(d0, d1, d2, d3, C0, R, S, pad, stride)) != B2B_OK) return st;
      if (kind == 2 && (st = check_channels(C1, 256)) != B2B_OK) return st;
      mode = kind == 2 ? MODE_CHAIN : MODE_SINGLE;
      if (R == 1 && S == 1 && pad == 0 && stride == 1)
        ok = gemm_params(p, mode, false, static_cast<int64_t>(d0) * d1 * d2, d3, C0, C1, &smem, &r,
                         forced);
      else
        ok = conv_params(p, mode, d0, d1, d2, d3, C0, R, S, pad, C1, &smem, &r, forced, stride);
      break;
    }
    case 5:   // b2b_gemm3: M, K0, N0, N1, N2
      if ((st = check_channels(d1, kMaxReduction)) != B2B_OK) return st;
      if ((st = check_channels(d2, 256)) != B2B_OK) return st;
      if ((st = check_channels(d3, 256)) != B2B_OK) return st;
      if ((st = check_channels(static_cast<int32_t>(dims[4]), 256)) != B2B_OK) return st;
      mode = MODE_CHAIN3;
      ok = gemm3_params(p, dims[0], d1, d2, d3, static_cast<int32_t>(dims[4]), &smem, &r, forced);
      break;
    case 4: { // conv_relu_maxpool: N, H, W, Cin, Cout
      const int32_t Cout = static_cast<int32_t>(dims[4]);
      if (d0 > 0 && (d1 < 2 || d2 < 2)) return B2B_ERR_SHAPE;
      if ((st = check_conv_args(d0, d1, d2, d3, Cout, 3, 3, 1)) != B2B_OK) return st;
      mode = MODE_POOL;
      ok = conv_params(p, MODE_POOL, d0, d1, d2, d3, Cout, 3, 3, 1, 0, &smem, &r, forced);
      break;
    }
  }
  return ok ? B2B_OK : B2B_ERR_UNSUPPORTED;
}

}  // extern "C"

// ------------------------------------------------------------------------------------
// tile-graph cost model (Welder notes, "Scheduling policy": enumerate candidate tile
// graphs, keep those within the memory footprint -- here, the planner's feasible layouts --
// order them by their traffic, and profile only the best few)
// ------------------------------------------------------------------------------------
// Per layout, lower bounds in microseconds on one launch from each resource it streams
// through: HBM (the problem's irreducible bytes over the copy rate), L2 -> SM (the busiest
// CTA's TMA and bias bytes over one SM's ingress) and the tensor pipe (the busiest CTA's
// share of the FLOPs over one SM's share of the peak).  Rates measured on the GB300 (copy
// bandwidth, cuBLAS bf16, one SM's TMA ingress from L2 at 2070 MHz); the model assumes its
// 152 SMs.  The same model, written for reading, is gemm_conv_chains_gb300/tilegraph.py
// (`launch_bounds`, `rank`); tests hold the two to the same choices.
namespace {
constexpr double kModelHbmGBs = 6791.4, kModelTensorTF = 1951.4, kModelSmMHz = 2070.0;
constexpr double kModelL2BytesPerClk = 89.0, kModelTol = 0.02;
constexpr int32_t kModelSms = 152, kModelSteadyTiles = 3, kModelTopK = 3;
constexpr double kModelABox = 128.0 * 64.0 * 2.0;   // one 128-row x 64-element A box

struct ModelEval {
  double d[3];        // the three bounds, largest first
  int32_t n;          // tiles of the busiest CTA (or CTA pair)
  bool shallow;       // fewer than three ring stages
};

// The problem's FLOPs, irreducible bytes, bias bytes per CTA, filter rows R and W2 bytes,
// and each GEMM's FLOPs and N (the MMA's N, padded to 16).
struct ModelProblem {
  double flops, floor_bytes, bias_cta, w2 = 0.0;
  int64_t R = 1;
  int32_t N0 = 0;
  bool three = false;
  int ngemm = 0;
  double gflops[3] = {0.0, 0.0, 0.0};
  int32_t gn[3] = {0, 0, 0};
  void gemm(double f, double n) {
    gflops[ngemm] = f;
    gn[ngemm++] = static_cast<int32_t>(round_up(static_cast<uint32_t>(n), 16u));
  }
};

// Tensor-pipe cycles per MMA of 128 rows per SM are N / 2 at the bf16 peak; shorter MMAs
// take a floor (measured on the GB300, operands resident: M128 x N64 x K16 48 cycles, the
// pair's M256 x N64 x K16 43 cycles per SM's 128 rows; N >= 128 runs at the peak).  The
// factor by which a GEMM of this N takes longer than the peak allows:
double model_mma_factor(int32_t n, bool pair) {
  const double ideal = std::max(1.0, n / 2.0), floor = pair ? 43.0 : 48.0;
  return std::max(1.0, floor / ideal);
}

ModelProblem model_problem(int32_t kind, const int64_t* d, int32_t ndims) {
  ModelProblem m;
  const double e = 2.0;
  switch (kind) {
    case 0: {   // M, K0, N0, N1
      const double M = d[0], K0 = d[1], N0 = d[2], N1 = d[3];
      m.flops = 2.0 * M * (K0 * N0 + N0 * N1);
      m.gemm(2.0 * M * K0 * N0, std::min(N0, 256.0));
      m.gemm(2.0 * M * N0 * N1, N1);
      m.floor_bytes = e * (M * K0 + K0 * N0 + N0 * N1 + M * N1) + (N0 + N1) * e;
      m.bias_cta = (N0 + N1) * e;
      m.N0 = static_cast<int32_t>(d[2]);
      break;
    }
    case 1: {   // M, K, N
      const double M = d[0], K = d[1], N = d[2];
      m.flops = 2.0 * M * (K * N);
      m.gemm(m.flops, N);
      m.floor_bytes = e * (M * K + K * N + N + M * N);
      m.bias_cta = N * e;
      m.N0 = static_cast<int32_t>(d[2]);
      break;
    }
    case 2:
    case 3: {   // N, H, W, C, C0, R, S, pad[, C1][, stride]
      const int64_t st = plan_stride(kind, d, ndims);
      const int64_t Ho = std::max<int64_t>(0, (d[1] + 2 * d[7] - d[5]) / st + 1);
      const int64_t Wo = std::max<int64_t>(0, (d[2] + 2 * d[7] - d[6]) / st + 1);
      const double M = static_cast<double>(d[0] * Ho * Wo);
      const double C = d[3], C0 = d[4], RS = static_cast<double>(d[5] * d[6]);
      const double C1 = kind == 2 ? static_cast<double>(d[8]) : 0.0;
      const double x = static_cast<double>(d[0] * d[1] * d[2]) * C;
      m.flops = 2.0 * M * (RS * C * C0 + C0 * C1);
      m.gemm(2.0 * M * RS * C * C0, C0);
      if (kind == 2) m.gemm(2.0 * M * C0 * C1, C1);
      m.floor_bytes = kind == 2 ? e * (x + C0 * RS * C + C0 + C1 * C0 + C1 + M * C1)
                                : e * (x + C0 * RS * C + C0 + M * C0);
      m.bias_cta = (C0 + C1) * e;
      m.R = d[5];
      m.N0 = static_cast<int32_t>(d[4]);
      break;
    }
    case 4: {   // N, H, W, Cin, Cout
      const double N = d[0], H = d[1], W = d[2], Cin = d[3], Cout = d[4];
      m.flops = 2.0 * N * H * W * 9.0 * Cin * Cout;
      m.gemm(m.flops, Cout);
      m.floor_bytes = e * (N * H * W * Cin + Cout * 9.0 * Cin + Cout +
                           N * static_cast<double>(d[1] / 2) * static_cast<double>(d[2] / 2) * Cout);
      m.bias_cta = Cout * e;
      m.R = 3;
      m.N0 = static_cast<int32_t>(d[4]);
      break;
    }
    default: {  // 5: M, K0, N0, N1, N2
      const double M = d[0], K0 = d[1], N0 = d[2], N1 = d[3], N2 = d[4];
      m.flops = 2.0 * M * (K0 * N0 + N0 * N1 + N1 * N2);
      m.gemm(2.0 * M * K0 * N0, N0);
      m.gemm(2.0 * M * N0 * N1, N1);
      m.gemm(2.0 * M * N1 * N2, N2);
      m.floor_bytes = e * (M * K0 + K0 * N0 + N0 * N1 + N1 * N2 + N0 + N1 + N2 + M * N2);
      m.bias_cta = (N0 + N1 + N2) * e;
      m.w2 = N1 * N2 * e;
      m.three = true;
      m.N0 = static_cast<int32_t>(d[2]);
      break;
    }
  }
  return m;
}

bool model_eval(int32_t kind, const int64_t* dims, int32_t ndims, int cand, ModelEval* out) {
  ChainParams p;
  Regions r;
  size_t smem = 0;
  int32_t mode = MODE_CHAIN;
  if (plan_for_kind(kind, dims, ndims, cand, p, r, smem, mode) != B2B_OK) return false;
  out->shallow = p.num_stages < 3u;
  if (p.num_tiles <= 0) {   // no work: nothing to order by
    out->d[0] = out->d[1] = out->d[2] = 0.0;
    out->n = 0;
    return true;
  }
  const ModelProblem m = model_problem(kind, dims, ndims);
  const double tiles = static_cast<double>(p.num_tiles);
  const double hbm = m.floor_bytes / (kModelHbmGBs * 1e3);
  double cta_bytes = 0.0, tensor = 0.0;
  int64_t n = 0;
  // the problem's MMA time at the peak rate, stretched for short MMAs
  double eff_flops = 0.0;
  for (int g = 0; g < m.ngemm; ++g)
    eff_flops += m.gflops[g] * model_mma_factor(m.gn[g], p.cta_pair != 0);
  const double sm_rate = kModelTensorTF * 1e6 / kModelSms;
  if (p.cta_pair && mode == MODE_POOL) {
    // conv + pool pairs: each CTA its own 8 x 16 tile of every pair-tile (halo boxes),
    // its half of the filters once, the bias of every channel once
    const int64_t pair_tiles = (p.num_tiles + 1) / 2;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(pair_tiles, kModelSms / 2));
    n = (pair_tiles + grid - 1) / grid;
    const double nn = static_cast<double>(n);
    cta_bytes = static_cast<double>(p.kstages0) * p.a_stage_bytes * nn +
                static_cast<double>(p.kchunks0) * p.w0_chunk_bytes + p.N0p * 2.0;
    tensor = eff_flops / tiles * nn / sm_rate;
  } else if (p.cta_pair) {
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(p.num_tiles, kModelSms / 2));
    n = (p.num_tiles + grid - 1) / grid;
    const double ctas = 2.0 * static_cast<double>(grid);
    const double A = tiles * 2.0 * p.kchunks0 * kModelABox;
    const double W0 = ctas * p.kchunks0 * p.w0_chunk_bytes;
    const double W1 = ctas * p.kchunks1 * p.w1_chunk_bytes;
    const double bias = ctas * (p.N0p / 2 + p.N1p / 2) * 2.0;
    cta_bytes = A / (2.0 * tiles) * static_cast<double>(n) + (W0 + W1 + bias) / ctas;
    tensor = eff_flops / (2.0 * tiles) * static_cast<double>(n) / sm_rate;
  } else {
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(p.num_tiles, kModelSms));
    const int64_t q = p.num_tiles / grid, rem = p.num_tiles % grid;
    n = q + (rem > 0 ? 1 : 0);
    const double ctas = static_cast<double>(grid);
    // W1 loads when grouped: once per pair of each CTA's tiles
    const double loads = static_cast<double>(rem * ((q + 2) / 2) + (grid - rem) * ((q + 1) / 2));
    double a_tile = p.halo ? static_cast<double>(p.kchunks0 / m.R) * p.a_stage_bytes
                           : p.kchunks0 * kModelABox;
    double w0 = static_cast<double>(p.kchunks0) * p.w0_chunk_bytes;
    if (p.p_split) {
      a_tile *= 2.0;
      const int32_t n0blk = (p.N0p + 63) / 64;
      const double hi = m.N0 % 64 == 0 ? static_cast<double>(p.w0_chunk_bytes) : (n0blk - 4) * 8192.0;
      w0 = p.kchunks0 * (p.w0_chunk_bytes + hi);
    }
    const double A = tiles * a_tile;
    const double w1 = static_cast<double>(p.kchunks1) * p.w1_chunk_bytes;
    const double bias = ctas * m.bias_cta;
    const double W2 = m.three ? ctas * m.w2 : 0.0;
    const double nn = static_cast<double>(n);
    cta_bytes = A / tiles * nn + bias / ctas + W2 / ctas;
    // W0: once per CTA when resident (alone or with W1), else once per tile
    const double W0 = (p.resident || m.three || p.w0_res) ? ctas * w0 : tiles * w0;
    cta_bytes += (p.resident || m.three || p.w0_res) ? W0 / ctas : W0 / tiles * nn;
    if (w1 != 0.0 || p.w0_res || m.three) {
      if (p.resident || m.three) {
        cta_bytes += (ctas * w1) / ctas;
      } else if (p.w1_group) {
        cta_bytes += (loads * w1) / loads * static_cast<double>((n + 1) / 2);
      } else {
        cta_bytes += (tiles * w1) / tiles * nn;
      }
    }
    tensor = eff_flops / tiles * nn / sm_rate;
  }
  const double l2 = cta_bytes / (kModelL2BytesPerClk * kModelSmMHz);
  double d[3] = {hbm, l2, tensor};
  std::sort(d, d + 3, [](double a, double b) { return a > b; });
  std::memcpy(out->d, d, sizeof(d));
  out->n = static_cast<int32_t>(n);
  return true;
}

// Whether the model orders x and y by their bounds (both in the steady state, and some
// bound differs by more than the tolerance); *sign < 0 if x is better.
bool model_orders(const ModelEval& x, const ModelEval& y, int* sign) {
  if (std::min(x.n, y.n) < kModelSteadyTiles) return false;
  for (int j = 0; j < 3; ++j) {
    const double a = x.d[j], b = y.d[j];
    if (std::fabs(a - b) > kModelTol * std::max(a, b)) {
      *sign = a < b ? -1 : 1;
      return true;
    }
  }
  return false;
}

// Steady state (both plans give their busiest CTA kModelSteadyTiles or more tiles): the
// bounds describe the launch, so the lower demand wins, resource by resource from the
// binding one.  Otherwise, or on a tie, the planner's order of preference stands (more
// tiles in flight, resident weights, separate staging; rings of three or more stages
// first): below the steady state a launch is mostly pipeline fill and drain, which the
// bounds do not see.
int model_compare(const ModelEval& x, int xi, const ModelEval& y, int yi) {
  int sign = 0;
  if (model_orders(x, y, &sign)) return sign;
  if (x.shallow != y.shallow) return x.shallow ? 1 : -1;
  return (xi > yi) - (xi < yi);
}

// Every feasible layout of a problem, best first.
b2b_status model_ranking(int32_t kind, const int64_t* dims, int32_t ndims,
                         std::vector<int32_t>* ranked) {
  ChainParams p;
  Regions r;
  size_t smem = 0;
  int32_t mode = MODE_CHAIN;
  if (b2b_status st = plan_for_kind(kind, dims, ndims, 0, p, r, smem, mode); st != B2B_OK)
    return st;
  std::vector<int32_t> left;
  std::vector<ModelEval> ev;
  for (int32_t c = 0; c < r.ncand; ++c) {
    ModelEval e;
    if (!model_eval(kind, dims, ndims, c, &e)) return B2B_ERR_UNSUPPORTED;
    left.push_back(c);
    ev.push_back(e);
  }
  ranked->clear();
  while (!left.empty()) {
    size_t best = 0;
    for (size_t i = 1; i < left.size(); ++i)
      if (model_compare(ev[i], left[i], ev[best], left[best]) < 0) best = i;
    ranked->push_back(left[best]);
    left.erase(left.begin() + static_cast<std::ptrdiff_t>(best));
    ev.erase(ev.begin() + static_cast<std::ptrdiff_t>(best));
  }
  return B2B_OK;
}

std::mutex g_model_mu;
std::map<std::vector<int64_t>, std::vector<int32_t>> g_model_top;   // by sizes
}  // namespace

// The top layouts of the model's ranking for a call's key (kind, sizes, variant): the best
// kModelTopK, then every later one the bounds do not order against the last of them (the
// model cannot tell those apart, so the profiler should).  Ranks by repeated selection of
// the best remaining layout, in the planner's order.
static b2b_status model_top(const std::vector<int64_t>& key, std::vector<int32_t>* top) {
  std::vector<int64_t> sizes(key.begin(), key.end() - 1);
  {
    std::lock_guard<std::mutex> lk(g_model_mu);
    const auto it = g_model_top.find(sizes);
    if (it != g_model_top.end()) {
      *top = it->second;
      return B2B_OK;
    }
  }
  const int32_t kind = static_cast<int32_t>(sizes[0]);
  const int64_t* dims = sizes.data() + 1;
  const int32_t ndims = static_cast<int32_t>(sizes.size()) - 1;
  std::vector<int32_t> ranked;
  if (b2b_status st = model_ranking(kind, dims, ndims, &ranked); st != B2B_OK) return st;
  std::vector<ModelEval> ev(ranked.size());
  for (size_t i = 0; i < ranked.size(); ++i) model_eval(kind, dims, ndims, ranked[i], &ev[i]);
  std::vector<int32_t> out;
  for (size_t i = 0; i < ranked.size(); ++i) {
    int sign = 0;
    if (static_cast<int>(i) >= kModelTopK &&
        model_orders(ev[kModelTopK - 1], ev[i], &sign))
      break;
    out.push_back(ranked[i]);
  }
  {
    std::lock_guard<std::mutex> lk(g_model_mu);
    g_model_top[sizes] = out;
  }
  *top = std::move(out);
  return B2B_OK;
}

extern "C" {

static b2b_status debug_plan_with(int32_t kind, const int64_t* dims, int32_t ndims, int forced,
                                  const Choice& c, uint32_t* out, int32_t out_len) {
  if (out == nullptr) return B2B_ERR_NULL;
  if (out_len < 64) return B2B_ERR_SHAPE;
  ChainParams p;
  Regions r;
  size_t smem = 0;
  int32_t mode = MODE_CHAIN;
  if (b2b_status st = plan_for_kind(kind, dims, ndims, forced, p, r, smem, mode); st != B2B_OK)
    return st;
  const uint32_t v[64] = {static_cast<uint32_t>(smem), p.num_stages, p.stage_bytes,
                          static_cast<uint32_t>(p.resident), static_cast<uint32_t>(p.out_alias_p),
                          p.off_ring, r.ring, p.off_w0, p.off_w1, r.w_res, p.w0_chunk_bytes,
                          p.w1_chunk_bytes, p.off_p[0], p.off_p[1], r.p_each, p.off_out[0],
                          p.off_out[1], r.out_each, p.off_bias, r.bias, p.off_bar, r.bar,
                          p.tmem_cols, p.d0_col[0], p.d0_col[1], p.d1_col[0], p.d1_col[1],
                          static_cast<uint32_t>(p.acc_dual), static_cast<uint32_t>(p.epi_groups),
                          static_cast<uint32_t>(p.num_tiles), static_cast<uint32_t>(p.kchunks0),
                          static_cast<uint32_t>(p.kchunks1), static_cast<uint32_t>(p.N0p),
                          static_cast<uint32_t>(p.N1p), static_cast<uint32_t>(mode),
                          static_cast<uint32_t>(p.p_tmem), static_cast<uint32_t>(p.w1_group),
                          p.w1_per_stage, static_cast<uint32_t>(p.halo), p.a_stage_bytes,
                          mode == MODE_POOL && p.cta_pair && p.two_issuers == 2 ? 6u
                                                                              : 1u << p.nbuf_log2,
                          p.off_p[2], p.off_p[3], p.d0_col[2], p.d0_col[3],
                          p.d1_col[2], p.d1_col[3], static_cast<uint32_t>(r.cand),
                          static_cast<uint32_t>(r.ncand), static_cast<uint32_t>(c.grid),
                          static_cast<uint32_t>(c.pf2), r.extend, p.off_w2, p.off_p1[0],
                          p.off_p1[1], p.d2_col[0], p.d2_col[1], p.p_split,
                          static_cast<uint32_t>(p.w0_res), static_cast<uint32_t>(p.cta_pair),
                          static_cast<uint32_t>(p.two_issuers),
                          static_cast<uint32_t>(p.out_slots), p.pt_col[0], p.pt_col[1]};
  std::memcpy(out, v, sizeof(v));
  return B2B_OK;
}

b2b_status b2b_debug_plan(int32_t kind, const int64_t* dims, int32_t ndims, uint32_t* out,
                          int32_t out_len) {
  b2b_status st = check_plan_args(kind, dims, ndims);
  if (st != B2B_OK) return st;
  const TuneKey key = plan_key(kind, dims, ndims);
  Choice c;
  if (!find_choice(key, &c) || c.cand < 0) {
    std::vector<int32_t> top;
    if ((st = model_top(key, &top)) != B2B_OK) return st;
    c.cand = top[0];
  }
  return debug_plan_with(kind, dims, ndims, c.cand, c, out, out_len);
}

b2b_status b2b_debug_plan_candidate(int32_t kind, const int64_t* dims, int32_t ndims,
                                    int32_t cand, uint32_t* out, int32_t out_len) {
  b2b_status st = check_plan_args(kind, dims, ndims);
  if (st != B2B_OK) return st;
  if (cand < 0) return B2B_ERR_SHAPE;
  return debug_plan_with(kind, dims, ndims, cand, Choice{cand, -1, -1}, out, out_len);
}

b2b_status b2b_set_choice(int32_t kind, const int64_t* dims, int32_t ndims, int32_t cand,
                          int32_t grid, int32_t prefetch_second) {
  b2b_status st = check_plan_args(kind, dims, ndims);
  if (st != B2B_OK) return st;
  if (cand < -1 || grid < -1 || grid > 2 || prefetch_second < -1 || prefetch_second > 1)
    return B2B_ERR_SHAPE;
  ChainParams p;
  Regions r;
  size_t smem = 0;
  int32_t mode = MODE_CHAIN;
  if ((st = plan_for_kind(kind, dims, ndims, cand, p, r, smem, mode)) != B2B_OK) return st;
  std::lock_guard<std::mutex> lk(g_tune_mu);
  Tuned& t = g_tuned[plan_key(kind, dims, ndims)];
  t = Tuned{};
  t.c = Choice{cand, grid, prefetch_second};
  t.source = 1;
  t.seq = ++g_tune_seq;
  return B2B_OK;
}

b2b_status b2b_get_choice(int32_t kind, const int64_t* dims, int32_t ndims, int32_t* out,
                          int32_t out_len) {
  b2b_status st = check_plan_args(kind, dims, ndims);
  if (st != B2B_OK) return st;
  if (out == nullptr) return B2B_ERR_NULL;
  if (out_len < 7) return B2B_ERR_SHAPE;
  Tuned t;
  {
    std::lock_guard<std::mutex> lk(g_tune_mu);
    if (const Tuned* f = find_for_query(plan_key(kind, dims, ndims))) t = *f;
  }
  const int32_t v[7] = {t.source, t.c.cand, t.c.grid, t.c.pf2, static_cast<int32_t>(t.best_ns),
                        static_cast<int32_t>(t.default_ns), static_cast<int32_t>(t.timed)};
  std::memcpy(out, v, sizeof(v));
  return B2B_OK;
}

b2b_status b2b_set_candidates(int32_t kind, const int64_t* dims, int32_t ndims,
                              const int32_t* cands, int32_t n) {
  b2b_status st = check_plan_args(kind, dims, ndims);
  if (st != B2B_OK) return st;
  if (cands == nullptr) return B2B_ERR_NULL;
  if (n < 1 || n > 64) return B2B_ERR_SHAPE;
  std::vector<int32_t> list;
  for (int32_t i = 0; i < n; ++i) {
    if (cands[i] < 0) return B2B_ERR_SHAPE;
    for (int32_t c : list)
      if (c == cands[i]) return B2B_ERR_SHAPE;
    ChainParams p;
    Regions r;
    size_t smem = 0;
    int32_t mode = MODE_CHAIN;
    if ((st = plan_for_kind(kind, dims, ndims, cands[i], p, r, smem, mode)) != B2B_OK) return st;
    list.push_back(cands[i]);
  }
  std::lock_guard<std::mutex> lk(g_tune_mu);
  Tuned& t = g_tuned[plan_key(kind, dims, ndims)];
  t = Tuned{};
  t.c = Choice{list[0], -1, -1};
  t.source = 3;
  t.seq = ++g_tune_seq;
  t.cands = std::move(list);
  return B2B_OK;
}

b2b_status b2b_get_tune_record(int32_t kind, const int64_t* dims, int32_t ndims, int32_t* out,
                               int32_t max_rows, int32_t* rows) {
  b2b_status st = check_plan_args(kind, dims, ndims);
  if (st != B2B_OK) return st;
  if (rows == nullptr || (out == nullptr && max_rows > 0)) return B2B_ERR_NULL;
  if (max_rows < 0) return B2B_ERR_SHAPE;
  std::lock_guard<std::mutex> lk(g_tune_mu);
  const Tuned* t = find_for_query(plan_key(kind, dims, ndims));
  const int32_t total = t ? static_cast<int32_t>(t->record.size()) : 0;
  *rows = total;
  for (int32_t i = 0; i < total && i < max_rows; ++i) {
    const TimedChoice& c = t->record[static_cast<size_t>(i)];
    const int32_t v[5] = {c.cand, c.grid, c.ctas, c.pf2, c.ns};
    std::memcpy(out + 5 * i, v, sizeof(v));
  }
  return B2B_OK;
}

void b2b_set_autotune(int32_t on) { g_autotune.store(on != 0 ? 1 : 0); }

void b2b_autotune_reset(void) {
  std::lock_guard<std::mutex> lk(g_tune_mu);
  g_tuned.clear();
}

b2b_status b2b_probe_timeout(uint64_t limit_ns, void* stream) {
  b2b_status st = B2B_OK;
  DeviceState* d = device_state(&st);
  if (d == nullptr) return st;
  if (limit_ns == 0 || limit_ns > 10000000000ull) return B2B_ERR_SHAPE;
  if (launch_probe_timeout(limit_ns, d->err, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return B2B_ERR_CUDA;
  }
  return B2B_OK;
}

}  // extern "C"
