// Packed attention forward on the sm_103a tensor cores, bf16 in and out,
// head_dim 64 (page "Source code for gigl.nn.packed_attention": every sequence
// attends only to itself within its cu_seqlens bounds; the op returns the
// output and the log-sum-exp).
//
// Design (one persistent CTA per SM, 12 warps):
//   warp 0      TMA producer: claims work items from the longest-first tile
//               plan, publishes them to a two-slot ring in shared memory, and
//               streams Q tiles and K/V blocks of 128 rows x 64 into a
//               four-stage ring with 128-byte swizzle.
//   warp 1      issues S_t = Q_t K_j^T (M=128, N=128, K=64) for both query
//               tiles into TMEM as soon as the softmax has read S_t of the
//               previous block, so the next scores are computed during this
//               block's softmax (warp 1 also owns tensor memory).
//   warps 2, 3  issue O_t += P_t V_j (M=128, N=64, K=128) for tile 0 and tile
//               1, P_t read from TMEM, when P_t(j) arrives.
//               A thread issues at most one MMA per ~130 cycles whatever its
//               size, and a block needs 4 QK and 8 PV MMAs per tile, so issue
//               is spread over three warps (whole warps, elect.sync) that each
//               commit their own completion barriers.
//   warps 4-7   softmax for query tile 0; warps 8-11 for query tile 1. Each
//               thread owns one query row (one TMEM lane): online softmax in
//               base 2 with fp32 statistics, P written back to TMEM as bf16,
//               O rescaled in TMEM when the row maximum grows, and the
//               epilogue (normalise, store the real rows, log-sum-exp).
// A work item is (sequence, head, pair of 128-row query tiles); both tiles
// share every K/V block, and while one tile's softmax runs the tensor cores
// work on the other tile. A sequence of at most 128 tokens has a single query
// tile, so (without a window) its items take two heads instead: tile t runs
// head h + t against its own K/V block, and both softmax warpgroups work. A
// sequence of at most 64 tokens packs two heads into each tile as well (rows
// 0-63 one head, rows 64-127 the next, loaded as 64-row boxes; each row masks
// the other head's half of the key columns), so an item takes four heads. A
// longer sequence with an odd number of 128-row blocks would end each head
// with an item of one tile; without a window those last tiles of two heads
// share an item instead, each tile against its own head's key blocks (which
// alternate in the K/V ring). With local attention (a window of key positions
// around each query position) an item visits only the key blocks its rows can
// see, and the softmax masks each row to its window. Keys past the sequence end are masked to -inf;
// query rows past it are computed but never stored. TMA zero-fills rows
// beyond the packed buffer.
//
// Tensor memory (512 columns): S0 [0,128) S1 [128,256) P0 [256,320)
// P1 [320,384) O0 [384,448) O1 [448,512).
//
// Every wait is bounded: after two seconds the CTA raises an abort flag,
// records PE_ERR_DEVICE_TIMEOUT in the workspace status word, drains its own
// copies and MMAs, frees tensor memory and exits.
#include <cudaTypedefs.h>

#include "pe_kernels.cuh"
#include "pe_sm103.cuh"

namespace pe {

namespace {

using namespace sm103;

constexpr int kRows = 128;                         // query rows per tile = keys per block
constexpr int kD = 64;                             // head_dim
constexpr int kStages = 4;                         // K/V ring depth
constexpr int kIssueWarps = 3;                     // QK issuer + one PV issuer per tile
constexpr int kThreads = 384;
// Registers per thread: 168 at launch (one CTA of 384 threads per SM); the
// producer/issuer warpgroup drops to kRegsLow and the two softmax warpgroups
// rise to kRegsHigh.
constexpr uint32_t kRegsLaunch = 168;
constexpr uint32_t kRegsLow = 56, kRegsHigh = 224;
static_assert(128 * (kRegsLow + 2 * kRegsHigh) <= kThreads * kRegsLaunch,
              "register split exceeds the launch allocation");
constexpr uint32_t kTileBytes = kRows * kD * 2;    // 16 KiB
constexpr int kPairRows = 2 * kRows;               // query rows per work item

// Tensor-memory column of S_t, P_t (bf16 pairs) and O_t for query tile t.
__host__ __device__ constexpr uint32_t col_s(int t) { return 128u * t; }
__host__ __device__ constexpr uint32_t col_p(int t) { return 256u + 64u * t; }
__host__ __device__ constexpr uint32_t col_o(int t) { return 384u + 64u * t; }
constexpr uint32_t kTmemCols = 512;

// Heads of a work item: one (kOneHead), one per tile (kHeadPerTile: tile t runs
// head + t), two per tile (kTwoHeadsPerTile: tile t runs head + 2t in rows
// 0-63 and head + 2t + 1 in rows 64-127), or the last query tiles of two heads
// of a longer sequence whose last pair would hold only one tile (kTailPair:
// tile t runs head + t over query rows pair*256 .., against key blocks of its
// own head, which alternate with the other tile's in the K/V ring).
enum : int32_t { kOneHead = 0, kHeadPerTile = 1, kTwoHeadsPerTile = 2, kTailPair = 3 };
struct Item {
  int32_t seq, head, pair;
  int32_t multi;
};
constexpr uint32_t kHalfTileBytes = kTileBytes / 2;  // 64 rows
// Output staging: the 32 rows of a softmax warp (4 KiB), 128-byte swizzled,
// written to HBM by one TMA store.
constexpr uint32_t kStageWarpBytes = 32 * kD * 2;

// kQSlots sets of the two Q tiles. With two (local attention, whose items
// are a few key blocks each) the next item's Q loads while this item's last
// QK products are still to be issued; full attention keeps one set.
template <int kQSlots>
struct alignas(1024) Smem {
  __nv_bfloat16 q[kQSlots][2][kRows * kD];
  __nv_bfloat16 k[kStages][kRows * kD];
  __nv_bfloat16 v[kStages][kRows * kD];
  alignas(1024) uint8_t ostage[8][kStageWarpBytes];   // per softmax warp, on the way to HBM
  uint64_t item_full[2], item_empty[2];
  uint64_t q_full[kQSlots], q_empty[kQSlots];
  uint64_t k_full[kStages], v_full[kStages], k_empty[kStages], v_empty[kStages];
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2], o_full[2];
  uint64_t drain[kIssueWarps];
  Item items[2];
  uint32_t tmem_base;
  WaitGuard guard;
};

// Plus the runtime 1024-byte alignment pad, within the 227 KiB a block may use.
static_assert(sizeof(Smem<2>) + 1024 <= 227 * 1024, "shared memory per block");
template <bool kLocal>
using FwdSmem = Smem<kLocal ? 2 : 1>;

struct FwdParams {
  const int32_t* cu;
  int32_t B, H;
  int32_t pair_heads_rows;  // sequences up to this long run a head per tile (0: never)
  int32_t quad_heads_rows;  // ... and up to this long two heads per tile (0: never)
  int32_t pair_odd_tails;   // longer sequences with an odd block count end in kTailPair items
  float scale_log2;
  __nv_bfloat16* out;
  float* lse;
  int64_t lse_stride;
  TilePlan plan;
  Window win;
  DeviceStatus* status;
  uint64_t wait_limit_ns;   // bounded-wait limit of this launch
};

// Where a wait gave up (recorded in the status word's detail field).
enum WaitSite { kSiteProducer = 1, kSiteMma = 2, kSiteSoftmax = 3 };

// The key blocks of an item: nkv blocks of 128 keys starting at key position
// kb0, and the blocks lo[t], lo[t] + step, ..., hi[t] that query tile t uses.
// Without a window that is the whole sequence for both tiles. With one, the
// blocks start at the first key of the item's window band (TMA rows need no
// alignment) and each tile uses only the blocks its own rows can see. A
// kTailPair item alternates the two heads' blocks (step 2).
struct ItemRange {
  int32_t kb0, nkv, lo0, hi0, lo1, hi1;   // (lo0, hi0) for tile 0, (lo1, hi1) for tile 1
  int32_t step;
  __device__ int32_t lo(int t) const { return t ? lo1 : lo0; }
  __device__ int32_t hi(int t) const { return t ? hi1 : hi0; }
  __device__ bool uses(int t, int32_t j) const {
    return j >= lo(t) && j <= hi(t) && (step == 1 || ((j - lo(t)) & 1) == 0);
  }
};

// Query tiles of an item.
__device__ __forceinline__ int item_tiles(const FwdParams& p, const Item& it, int32_t len) {
  if (it.multi == kHeadPerTile || it.multi == kTailPair) return 2;
  if (it.multi == kTwoHeadsPerTile) return p.H - it.head > 2 ? 2 : 1;
  return len - it.pair * kPairRows > kRows ? 2 : 1;
}

template <bool kLocal>
__device__ __forceinline__ ItemRange item_range(const FwdParams& p, int32_t len, int32_t r0,
                                                int32_t multi, int ntiles) {
  ItemRange ir;
  ir.step = 1;
  if (multi == kTailPair) {  // block j: keys 128*(j/2) .. of tile (j & 1)'s head
    const int32_t nb = (len + kRows - 1) / kRows;
    ir.kb0 = 0;
    ir.nkv = 2 * nb;
    ir.lo0 = 0;
    ir.hi0 = 2 * nb - 2;
    ir.lo1 = 1;
    ir.hi1 = 2 * nb - 1;
    ir.step = 2;
    return ir;
  }
  if (multi != kOneHead) {  // block j holds the keys of tile j's heads and serves it only
    ir.kb0 = 0;
    ir.nkv = ntiles;
    ir.lo0 = ir.hi0 = 0;
    ir.lo1 = 1;
    ir.hi1 = ntiles - 1;
    return ir;
  }
  if (!kLocal) {
    ir.kb0 = 0;
    ir.nkv = (len + kRows - 1) / kRows;
    ir.lo0 = ir.lo1 = 0;
    ir.hi0 = ir.hi1 = ir.nkv - 1;
    return ir;
  }
  ir.kb0 = window_lo(p.win, r0);
  const int32_t last = min(r0 + kPairRows, len) - 1;
  ir.nkv = (window_hi(p.win, last, len) - ir.kb0) / kRows + 1;
  ir.lo0 = 0;                        // tile 0 starts the band
  ir.hi0 = (window_hi(p.win, min(r0 + kRows, len) - 1, len) - ir.kb0) / kRows;
  if (r0 + kRows < len) {
    ir.lo1 = (window_lo(p.win, r0 + kRows) - ir.kb0) / kRows;
    ir.hi1 = ir.nkv - 1;             // tile 1 ends it
  } else {                           // no tile 1 in this item
    ir.lo1 = 1;
    ir.hi1 = 0;
  }
  return ir;
}

__device__ __forceinline__ void decode_item(const FwdParams& p, int32_t t, Item& it) {
  int32_t seq, local;
  plan_decode(p.plan.order, p.plan.tile_end, p.B, t, seq, local);
  const int32_t len = __ldg(p.cu + seq + 1) - __ldg(p.cu + seq);
  it.seq = seq;
  it.pair = 0;
  if (len <= p.quad_heads_rows) {  // local indexes groups of four heads
    it.head = 4 * local;
    it.multi = kTwoHeadsPerTile;
    return;
  }
  if (len <= p.pair_heads_rows) {  // local indexes pairs of heads
    it.head = 2 * local;
    it.multi = it.head + 1 < p.H ? kHeadPerTile : kOneHead;
    return;
  }
  const int32_t npairs = (len + kPairRows - 1) / kPairRows;
  if (p.pair_odd_tails && (((len + kRows - 1) / kRows) & 1)) {
    // The heads' full pairs first, then their last tiles two heads at a time.
    const int32_t full = npairs - 1;
    if (local < p.H * full) {
      it.head = local / full;
      it.pair = local - it.head * full;
      it.multi = kOneHead;
      return;
    }
    it.head = 2 * (local - p.H * full);
    it.pair = full;
    it.multi = it.head + 1 < p.H ? kTailPair : kOneHead;
    return;
  }
  it.head = local / npairs;
  it.pair = local - it.head * npairs;
  it.multi = kOneHead;
}

// Head loaded into half hh (rows 64*hh ..) of tile (or block) t of a
// two-heads-per-tile item; a missing last head repeats the tile's first head,
// whose rows there are computed but never stored.
__device__ __forceinline__ int32_t packed_head(const FwdParams& p, const Item& it, int t, int hh) {
  const int32_t h = it.head + 2 * t + hh;
  return h < p.H ? h : it.head + 2 * t;
}

// kLocal selects the local-attention variant (window masks, block ranges and
// the guard for rows that have seen no visible key); full attention compiles
// without any of it.
template <bool kLocal>
__global__ void __launch_bounds__(kThreads, 1)
fwd_sm103_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v,
                 const __grid_constant__ CUtensorMap tm_q64,
                 const __grid_constant__ CUtensorMap tm_k64,
                 const __grid_constant__ CUtensorMap tm_v64,
                 const __grid_constant__ CUtensorMap tm_o, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  constexpr int kQSlots = kLocal ? 2 : 1;
  FwdSmem<kLocal>& S =
      *reinterpret_cast<FwdSmem<kLocal>*>(smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile WaitGuard* abort_flag = &S.guard;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&S.item_full[i]), 1);
      mbar_init(smem_u32(&S.item_empty[i]), kIssueWarps + 8);
      mbar_init(smem_u32(&S.s_full[i]), 1);
      mbar_init(smem_u32(&S.s_free[i]), 4);
      mbar_init(smem_u32(&S.pv_done[i]), 1);
      mbar_init(smem_u32(&S.p_full[i]), 4);
      mbar_init(smem_u32(&S.o_full[i]), 1);
    }
    for (int i = 0; i < kQSlots; ++i) {
      mbar_init(smem_u32(&S.q_full[i]), 1);
      mbar_init(smem_u32(&S.q_empty[i]), 1);       // the QK issuer, after an item's last QK
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&S.k_full[s]), 1);
      mbar_init(smem_u32(&S.v_full[s]), 1);
      mbar_init(smem_u32(&S.k_empty[s]), 1);       // the QK issuer, after both tiles' QK
      mbar_init(smem_u32(&S.v_empty[s]), 2);       // each PV issuer, once per block
    }
    for (int w = 0; w < kIssueWarps; ++w) mbar_init(smem_u32(&S.drain[w]), 1);
    S.guard.abort = 0;
    S.guard.limit_ns = p.wait_limit_ns;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&S.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = __shfl_sync(0xffffffffu, S.tmem_base, 0);
  // Launched behind the tile plan: read it (and the status word) only once
  // that kernel has finished.
  griddep_wait();
  const int32_t total = *p.plan.total_tiles;

  // Warpgroup 0 (TMA producer, MMA issuers) hands registers to the two
  // softmax warpgroups; each warpgroup's setmaxnreg heads its own branch.
  if (warp < 4) {
    regs_release<kRegsLow>();
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        uint32_t kv_no = 0;
        int pending_q[kQSlots];            // per Q slot: parity of the last load not yet known complete
        for (int i = 0; i < kQSlots; ++i) pending_q[i] = -1;
        int pending_k[kStages], pending_v[kStages];  // parity of the last K / V load per stage
        for (int s = 0; s < kStages; ++s) pending_k[s] = pending_v[s] = -1;
        bool ok = true;
        for (uint32_t item_no = 0; ok; ++item_no) {
          const int slot = item_no & 1;
          if (!mbar_wait(smem_u32(&S.item_empty[slot]), ((item_no >> 1) & 1) ^ 1, abort_flag,
                         p.status, kSiteProducer)) {
            ok = false;
            break;
          }
          const int32_t t = atomicAdd(p.plan.counter, 1);
          Item it;
          if (t >= total) {
            it.seq = -1;
            it.head = it.pair = it.multi = 0;
          } else {
            decode_item(p, t, it);
          }
          S.items[slot] = it;
          mbar_arrive(smem_u32(&S.item_full[slot]));
          if (it.seq < 0) break;
          const int32_t start = __ldg(p.cu + it.seq);
          const int32_t len = __ldg(p.cu + it.seq + 1) - start;
          const int32_t r0 = it.pair * kPairRows;
          const int ntiles = item_tiles(p, it, len);
          const ItemRange ir = item_range<kLocal>(p, len, r0, it.multi, ntiles);
          const int32_t nkv = ir.nkv;
          const int32_t x = it.head * kD;
          // Q slot qs was last read by the QK products of item item_no - kQSlots.
          const int qs = item_no % kQSlots;
          const uint32_t q_par = (item_no / kQSlots) & 1;
          if (!mbar_wait(smem_u32(&S.q_empty[qs]), q_par ^ 1, abort_flag, p.status,
                         kSiteProducer)) {
            ok = false;
            break;
          }
          const uint32_t q_bar = smem_u32(&S.q_full[qs]);
          mbar_arrive_expect_tx(q_bar, ntiles * kTileBytes);
          // Multi-head items load every tile (and K/V block) from the
          // sequence's first row: one head's columns per tile, or two heads'
          // in 64-row halves.
          for (int tt = 0; tt < ntiles; ++tt) {
            if (it.multi == kTwoHeadsPerTile) {
              for (int hh = 0; hh < 2; ++hh)
                tma_load_2d(smem_u32(S.q[qs][tt]) + hh * kHalfTileBytes, &tm_q64, q_bar,
                            packed_head(p, it, tt, hh) * kD, start);
            } else if (it.multi == kTailPair) {  // both tiles: rows r0.., heads head + tt
              tma_load_2d(smem_u32(S.q[qs][tt]), &tm_q, q_bar, x + tt * kD, start + r0);
            } else {
              tma_load_2d(smem_u32(S.q[qs][tt]), &tm_q, q_bar, it.multi ? x + tt * kD : x,
                          it.multi ? start : start + r0 + tt * kRows);
            }
          }
          pending_q[qs] = static_cast<int>(q_par);
          for (int32_t j = 0; j < nkv; ++j, ++kv_no) {
            const int s = kv_no % kStages;
            const uint32_t ph = (kv_no / kStages) & 1;
            if (!mbar_wait(smem_u32(&S.k_empty[s]), ph ^ 1, abort_flag, p.status, kSiteProducer)) {
              ok = false;
              break;
            }
            const bool packed = it.multi == kTwoHeadsPerTile;
            const bool tail = it.multi == kTailPair;
            const int32_t kx = tail ? x + (j & 1) * kD : (it.multi ? x + j * kD : x);
            const int32_t ky = tail ? start + (j >> 1) * kRows
                                    : (it.multi ? start : start + ir.kb0 + j * kRows);
            mbar_arrive_expect_tx(smem_u32(&S.k_full[s]), kTileBytes);
            if (packed) {
              for (int hh = 0; hh < 2; ++hh)
                tma_load_2d(smem_u32(S.k[s]) + hh * kHalfTileBytes, &tm_k64,
                            smem_u32(&S.k_full[s]), packed_head(p, it, j, hh) * kD, start);
            } else {
              tma_load_2d(smem_u32(S.k[s]), &tm_k, smem_u32(&S.k_full[s]), kx, ky);
            }
            pending_k[s] = (int)ph;
            if (!mbar_wait(smem_u32(&S.v_empty[s]), ph ^ 1, abort_flag, p.status, kSiteProducer)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(smem_u32(&S.v_full[s]), kTileBytes);
            if (packed) {
              for (int hh = 0; hh < 2; ++hh)
                tma_load_2d(smem_u32(S.v[s]) + hh * kHalfTileBytes, &tm_v64,
                            smem_u32(&S.v_full[s]), packed_head(p, it, j, hh) * kD, start);
            } else {
              tma_load_2d(smem_u32(S.v[s]), &tm_v, smem_u32(&S.v_full[s]), kx, ky);
            }
            pending_v[s] = (int)ph;
          }
        }
        if (!ok) {
          // Let every copy this thread started land before the CTA exits.
          for (int i = 0; i < kQSlots; ++i)
            if (pending_q[i] >= 0) mbar_drain_wait(smem_u32(&S.q_full[i]), (uint32_t)pending_q[i]);
          for (int s = 0; s < kStages; ++s) {
            if (pending_k[s] >= 0) mbar_drain_wait(smem_u32(&S.k_full[s]), (uint32_t)pending_k[s]);
            if (pending_v[s] >= 0) mbar_drain_wait(smem_u32(&S.v_full[s]), (uint32_t)pending_v[s]);
          }
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ QK issuer (whole warp)
      // S_t for key block j+1 is computed as soon as the softmax has read S_t(j),
      // so it overlaps that softmax.
      constexpr uint32_t idesc_qk = idesc_bf16(kRows, kRows, false, false);
      uint32_t kv_no = 0;
      uint32_t n_qk[2] = {0, 0};                     // QK MMA groups issued per tile, all items
      bool ok = true;
      for (uint32_t item_no = 0; ok; ++item_no) {
        const int slot = item_no & 1;
        if (!warp_wait(smem_u32(&S.item_full[slot]), (item_no >> 1) & 1, abort_flag, p.status,
                       kSiteMma))
          break;
        const Item it = S.items[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&S.item_empty[slot]));
        if (it.seq < 0) break;
        const int32_t len = __ldg(p.cu + it.seq + 1) - __ldg(p.cu + it.seq);
        const int32_t r0 = it.pair * kPairRows;
        const int ntiles = item_tiles(p, it, len);
        const ItemRange ir = item_range<kLocal>(p, len, r0, it.multi, ntiles);
        const int32_t nkv = ir.nkv;
        const int qs = item_no % kQSlots;
        if (!warp_wait(smem_u32(&S.q_full[qs]), (item_no / kQSlots) & 1, abort_flag, p.status,
                       kSiteMma))
          break;
        for (int32_t j = 0; j < nkv && ok; ++j) {
          const uint32_t c = kv_no + j;
          const int s = c % kStages;
          if (!warp_wait(smem_u32(&S.k_full[s]), (c / kStages) & 1, abort_flag, p.status,
                         kSiteMma)) {
            ok = false;
            break;
          }
          const uint32_t k_addr = smem_u32(S.k[s]);
          for (int t = 0; t < ntiles; ++t) {
            // Outside every window of tile t, or the other head's block.
            if ((kLocal || it.multi) && !ir.uses(t, j)) continue;
            // The softmax must have read the previous S_t before it is overwritten.
            if (n_qk[t] > 0 && !warp_wait(smem_u32(&S.s_free[t]), (n_qk[t] - 1) & 1, abort_flag,
                                          p.status, kSiteMma)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t q_addr = smem_u32(S.q[qs][t]);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              mma_ss_warp(tmem + col_s(t), smem_desc_sw128(q_addr + kk * 32, 16, 1024),
                          smem_desc_sw128(k_addr + kk * 32, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
            tc_commit_warp(smem_u32(&S.s_full[t]));
            ++n_qk[t];
          }
          if (!ok) break;
          tc_commit_warp(smem_u32(&S.k_empty[s]));  // K_j no longer needed by either tile
        }
        kv_no += nkv;
        if (ok) tc_commit_warp(smem_u32(&S.q_empty[qs]));
      }
      // Every MMA this warp issued must finish before tensor memory is freed.
      tc_commit_warp(smem_u32(&S.drain[0]));
      mbar_drain_wait(smem_u32(&S.drain[0]), 0);
    } else if (warp == 2 || warp == 3) {
      // ------------------------------------------------------------ PV issuers (whole warps)
      // O_t += P_t V_j as soon as the softmax has written P_t(j).
      const int t = warp - 2;
      constexpr uint32_t idesc_pv = idesc_bf16(kRows, kD, false, true);
      uint32_t kv_no = 0, n_pv = 0;
      bool ok = true;
      for (uint32_t item_no = 0; ok; ++item_no) {
        const int slot = item_no & 1;
        if (!warp_wait(smem_u32(&S.item_full[slot]), (item_no >> 1) & 1, abort_flag, p.status,
                       kSiteMma))
          break;
        const Item it = S.items[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&S.item_empty[slot]));
        if (it.seq < 0) break;
        const int32_t len = __ldg(p.cu + it.seq + 1) - __ldg(p.cu + it.seq);
        const int32_t r0 = it.pair * kPairRows;
        const int ntiles = item_tiles(p, it, len);
        const ItemRange ir = item_range<kLocal>(p, len, r0, it.multi, ntiles);
        const int32_t nkv = ir.nkv;
        for (int32_t j = 0; j < nkv; ++j) {
          const uint32_t c = kv_no + j;
          const int s = c % kStages;
          // Both PV warps take part in every V stage phase: each waits for every
          // block and releases it once, so the producer can never refill a stage
          // that either warp has not yet seen (which would make a parity wait
          // match a later phase).
          if (!warp_wait(smem_u32(&S.v_full[s]), (c / kStages) & 1, abort_flag, p.status,
                         kSiteMma)) {
            ok = false;
            break;
          }
          if (t >= ntiles || !ir.uses(t, j)) {       // this tile does not read V_j
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&S.v_empty[s]));
            continue;
          }
          if (!warp_wait(smem_u32(&S.p_full[t]), n_pv & 1, abort_flag, p.status, kSiteMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t v_addr = smem_u32(S.v[s]);
#pragma unroll
          for (int kk = 0; kk < kRows / 16; ++kk)
            mma_ts_warp(tmem + col_o(t), tmem + col_p(t) + kk * 8,
                        smem_desc_sw128(v_addr + kk * 16 * 128, 16, 1024), idesc_pv,
                        (j > ir.lo(t) || kk > 0) ? 1u : 0u);
          tc_commit_warp(smem_u32(&S.pv_done[t]));
          if (j == ir.hi(t)) tc_commit_warp(smem_u32(&S.o_full[t]));
          ++n_pv;
          tc_commit_warp(smem_u32(&S.v_empty[s]));
        }
        kv_no += nkv;
      }
      tc_commit_warp(smem_u32(&S.drain[1 + t]));
      mbar_drain_wait(smem_u32(&S.drain[1 + t]), 0);
    }
  } else {
    regs_claim<kRegsHigh>();
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;               // query tile of this warpgroup
    const int quarter = warp & 3;                // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;         // query row within the tile
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    uint32_t s_cnt = 0, o_cnt = 0;               // S blocks and items consumed by this tile
    const float scale_log2 = p.scale_log2;
    for (uint32_t item_no = 0;; ++item_no) {
      const int slot = item_no & 1;
      if (!warp_wait(smem_u32(&S.item_full[slot]), (item_no >> 1) & 1, abort_flag, p.status,
                     kSiteSoftmax))
        break;
      const Item it = S.items[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&S.item_empty[slot]));
      if (it.seq < 0) break;
      const int32_t start = __ldg(p.cu + it.seq);
      const int32_t len = __ldg(p.cu + it.seq + 1) - start;
      // Multi-head items: this tile runs head + t over the sequence's rows, or
      // (two heads per tile) head + 2t in rows 0-63 and head + 2t + 1 in rows
      // 64-127, each row seeing its own head's half of the key columns.
      const int ntiles = item_tiles(p, it, len);
      if (t >= ntiles) continue;                 // this tile of the item is empty
      const bool packed = it.multi == kTwoHeadsPerTile;
      const int32_t r0 = it.multi == kTailPair ? it.pair * kPairRows
                         : (it.multi ? 0 : it.pair * kPairRows + t * kRows);
      const int32_t head = packed ? it.head + 2 * t + (quarter >> 1)
                                  : (it.multi ? it.head + t : it.head);
      const int32_t pos = packed ? (row & 63) : r0 + row;   // this row's query position
      const int32_t coff = packed ? (quarter >> 1) * 64 : 0;  // column of key position 0
      const ItemRange ir = item_range<kLocal>(p, len, it.pair * kPairRows, it.multi, ntiles);
      // This row's visible key positions (local attention).
      const int32_t vis_lo = kLocal ? window_lo(p.win, r0 + row) : 0;
      const int32_t vis_hi = kLocal ? window_hi(p.win, r0 + row, len) : len - 1;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int32_t j = ir.lo(t); j <= ir.hi(t); j += ir.step) {
        const bool first_blk = j == ir.lo(t);
        if (!warp_wait(smem_u32(&S.s_full[t]), s_cnt & 1, abort_flag, p.status, kSiteSoftmax)) {
          ok = false;
          break;
        }
        ++s_cnt;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + col_s(t) + 32 * c, sr[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_wait_ld(sr[c]);
        // S_t is in registers: the next block's scores may overwrite it.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&S.s_free[t]));
        // Key position of column coff.
        const int32_t kb = it.multi == kTailPair ? (j >> 1) * kRows
                                                 : (it.multi ? 0 : ir.kb0 + j * kRows);
        const int32_t kv_valid = len - kb;         // > 0; columns at or past it are masked
        if (kLocal) {
          // Columns outside [vis_lo, vis_hi] (which also ends before len).
          const int32_t clo = vis_lo - kb, chi = vis_hi - kb;
          if (__any_sync(0xffffffffu, clo > 0 || chi < kRows - 1)) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (32 * c + e < clo || 32 * c + e > chi) sr[c][e] = 0xff800000u;  // -inf
          }
        } else if (kv_valid < kRows) {             // only a sequence's last key block
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (32 * c + e < coff || 32 * c + e >= coff + kv_valid) sr[c][e] = 0xff800000u;
        }
        // Row maximum of the raw scores (scale > 0 commutes with max), four
        // independent chains of 3-input max.
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; e += 8)
#pragma unroll
            for (int u = 0; u < 4; ++u)
              mx[u] = max3(mx[u], __uint_as_float(sr[c][e + 2 * u]),
                           __uint_as_float(sr[c][e + 2 * u + 1]));
        const float m_blk = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * scale_log2;
        // Lazy rescaling: the running maximum moves only when the block's
        // maximum exceeds it by more than 2^8; until then exponents stay <= 2^8.
        const bool grow = m_blk > m + 8.f;
        const float m_new = grow ? m_blk : m;
        const float alpha = grow ? ex2(m - m_new) : 1.f;  // 0 on the first block
        // Exponents first, into registers: the wait for P_t(j-1) V below then
        // hides behind this work instead of delaying it.
        // With a window a row may have seen no visible key yet (m_new = -inf):
        // its exponents are then taken against 0 and stay exactly 0. Without
        // one every block holds a visible key for every row.
        const float m_use = (kLocal && m_new == -INFINITY) ? 0.f : m_new;
        const uint64_t c2 = f2(scale_log2, scale_log2), nm2 = f2(-m_use, -m_use);
        uint64_t acc[4] = {0, 0, 0, 0};
        uint32_t pk[4][16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint64_t x = ffma2(f2(__uint_as_float(sr[c][2 * e]),
                                        __uint_as_float(sr[c][2 * e + 1])), c2, nm2);
            float p0, p1;
            f2_split(x, p0, p1);
            p0 = ex2(p0);
            p1 = ex2(p1);
            acc[e & 3] = fadd2(acc[e & 3], f2(p0, p1));
            pk[c][e] = pack_bf16x2(p0, p1);
          }
        }
        float s0, s1, s2, s3, s4, s5, s6, s7;
        f2_split(acc[0], s0, s1);
        f2_split(acc[1], s2, s3);
        f2_split(acc[2], s4, s5);
        f2_split(acc[3], s6, s7);
        l = l * alpha + (((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7)));
        m = m_new;
        if (!first_blk) {
          // P_t(j-1) V must have finished before P_t is overwritten or O_t rescaled.
          if (!warp_wait(smem_u32(&S.pv_done[t]), (s_cnt - 2) & 1, abort_flag, p.status,
                         kSiteSoftmax)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_st16(lane_base + col_p(t) + 16 * c, pk[c]);
        // O holds P(j-1) V(j-1): rescale it when some row's maximum moved.
        if (!first_blk && __any_sync(0xffffffffu, grow)) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t o[32];
            tmem_ld32(lane_base + col_o(t) + 32 * h, o);
            tmem_wait_ld(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(lane_base + col_o(t) + 32 * h, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&S.p_full[t]));
      }
      if (!ok) break;
      if (!warp_wait(smem_u32(&S.o_full[t]), o_cnt & 1, abort_flag, p.status, kSiteSoftmax))
        break;
      ++o_cnt;
      tc_fence_after();
      uint32_t o[2][32];
      tmem_ld32(lane_base + col_o(t), o[0]);
      tmem_ld32(lane_base + col_o(t) + 32, o[1]);
      tmem_wait_ld(o[0]);
      tmem_wait_ld(o[1]);
      // A warp's 32 rows are 32 consecutive tokens of one head: when all of
      // them are real they go through shared memory to one TMA store (the
      // copy engine moves 4 KiB, no 16-byte stores of 32 rows at a time from
      // the warp); the partial warp at a sequence's end stores its rows itself.
      const int32_t pos0 = pos - lane;                  // warp-uniform
      const bool real = pos < len && head < p.H;        // (a repeated head's rows are not stored)
      const float inv = 1.f / l;
      const int64_t tok = static_cast<int64_t>(start) + pos;
      if (head < p.H && len - pos0 >= 32) {
        uint8_t* stage = S.ostage[warp - 4];
        if (lane == 0) bulk_wait_read();                // the previous store has left the stage
        __syncwarp();
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const uint32_t* src = o[g >> 2] + (g & 3) * 8;
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(src[0]) * inv, __uint_as_float(src[1]) * inv);
          w.y = pack_bf16x2(__uint_as_float(src[2]) * inv, __uint_as_float(src[3]) * inv);
          w.z = pack_bf16x2(__uint_as_float(src[4]) * inv, __uint_as_float(src[5]) * inv);
          w.w = pack_bf16x2(__uint_as_float(src[6]) * inv, __uint_as_float(src[7]) * inv);
          *reinterpret_cast<uint4*>(stage + lane * 128 + ((g ^ (lane & 7)) << 4)) = w;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tm_o, smem_u32(stage), head * kD, start + pos0);
          bulk_commit();
        }
      } else if (real) {
        uint4* dst = reinterpret_cast<uint4*>(p.out + (tok * p.H + head) * kD);
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const uint32_t* src = o[g >> 2] + (g & 3) * 8;
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(src[0]) * inv, __uint_as_float(src[1]) * inv);
          w.y = pack_bf16x2(__uint_as_float(src[2]) * inv, __uint_as_float(src[3]) * inv);
          w.z = pack_bf16x2(__uint_as_float(src[4]) * inv, __uint_as_float(src[5]) * inv);
          w.w = pack_bf16x2(__uint_as_float(src[6]) * inv, __uint_as_float(src[7]) * inv);
          dst[g] = w;
        }
      }
      if (real && p.lse) p.lse[static_cast<int64_t>(head) * p.lse_stride + tok] =
          (m + __log2f(l)) * kLn2;
    }
    bulk_wait_all();                    // every row is written before the CTA retires
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

pe_status get_encoder() {
  if (g_encode) return PE_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult qres;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &qres) != cudaSuccess ||
      qres != cudaDriverEntryPointSuccess || !fn)
    return PE_ERR_CUDA;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return PE_OK;
}

// [N, H*64] bf16 rows; boxes of box_rows rows x 64 columns (one head), 128-byte
// swizzle (loads of q, k, v; stores of 32-row output boxes).
pe_status make_map(CUtensorMap* map, const void* base, int64_t N, int32_t H,
                   uint32_t box_rows = kRows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(H) * kD, static_cast<cuuint64_t>(N)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * kD * 2};
  cuuint32_t box[2] = {kD, box_rows};
  cuuint32_t elem_strides[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PE_OK : PE_ERR_CUDA;
}

}  // namespace

int sm103_fwd_rows_per_item() { return kPairRows; }
int sm103_fwd_pair_heads_rows(Window win) { return win.active() ? 0 : kRows; }
int sm103_fwd_quad_heads_rows(Window win) { return win.active() ? 0 : kRows / 2; }
int sm103_fwd_pair_odd_tails(Window win) { return win.active() ? 0 : 1; }

pe_status fwd_sm103(const void* q, const void* k, const void* v, const int32_t* cu, int32_t B,
                    int32_t H, int64_t N, float scale, Window win, void* out, float* lse,
                    TilePlan plan, DeviceStatus* status, cudaStream_t stream) {
  PE_TRY(get_encoder());
  CUtensorMap mq, mk, mv, mq64, mk64, mv64, mo;
  PE_TRY(make_map(&mo, out, N, H, 32));
  PE_TRY(make_map(&mq, q, N, H));
  PE_TRY(make_map(&mk, k, N, H));
  PE_TRY(make_map(&mv, v, N, H));
  PE_TRY(make_map(&mq64, q, N, H, 64));
  PE_TRY(make_map(&mk64, k, N, H, 64));
  PE_TRY(make_map(&mv64, v, N, H, 64));
  const size_t smem = (win.active() ? sizeof(FwdSmem<true>) : sizeof(FwdSmem<false>)) + 1024;
  auto kernel = win.active() ? fwd_sm103_kernel<true> : fwd_sm103_kernel<false>;
  PE_CUDA_TRY(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(smem)));
  // The softmax warpgroups' register claim is served from what the CTA was
  // launched with; never launch a build whose count cannot serve it.
  cudaFuncAttributes attr;
  PE_CUDA_TRY(cudaFuncGetAttributes(&attr, kernel));
  if (static_cast<uint32_t>(attr.numRegs) * kThreads < 128u * (kRegsLow + 2 * kRegsHigh))
    return PE_ERR_UNSUPPORTED;
  FwdParams prm;
  prm.cu = cu;
  prm.B = B;
  prm.H = H;
  prm.pair_heads_rows = sm103_fwd_pair_heads_rows(win);
  prm.quad_heads_rows = sm103_fwd_quad_heads_rows(win);
  prm.pair_odd_tails = sm103_fwd_pair_odd_tails(win);
  prm.scale_log2 = scale * kLog2e;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.lse = lse;
  prm.lse_stride = N;
  prm.plan = plan;
  prm.win = win;
  prm.status = status;
  prm.wait_limit_ns = wait_limit_ns();
  PE_TRY(launch_after_previous(kernel, dim3(device_sm_count()), dim3(kThreads), smem, stream, mq,
                               mk, mv, mq64, mk64, mv64, mo, prm));
  PE_CUDA_TRY(cudaGetLastError());
  return PE_OK;
}

}  // namespace pe
