// Packed attention forward on the sm_103a tensor cores, bf16 in and out,
// head_dim 128, full attention (page "Source code for gigl.nn.packed_attention":
// every sequence attends only to itself within its cu_seqlens bounds; the
// op returns the output and the log-sum-exp; "Constraints": any head_dim that
// is a multiple of 8).
//
// The head_dim-64 kernel's design with the tensor-memory plan that 128-wide
// outputs need: two query tiles' scores (2 x 128 columns) and outputs (2 x 128)
// fill the 512 columns, so each tile's P (bf16, 64 columns) is written over the
// first half of its own score columns once the softmax holds the scores in
// registers. QK of the tile's next block then waits until P V of this block has
// read P (and thereby until the softmax has read the scores); the softmax needs
// no wait before writing P or rescaling O, because the next scores can only
// exist once the previous P V has completed.
//
//   warp 0      TMA producer: claims work items from the longest-first plan and
//               streams Q tiles and K/V blocks (128 rows x 128 as two 64-column
//               boxes with 128-byte swizzle) into a two-stage ring.
//   warp 1      issues S_t = Q_t K_j^T (M=128, N=128, K=128: 8 MMAs) for both
//               query tiles.
//   warps 2, 3  issue O_t += P_t V_j for tile 0 and tile 1 (M=128, N=64 per
//               64-column half of V, K=128 keys: 16 MMAs).
//   warps 4-7   softmax of query tile 0, warps 8-11 of query tile 1: one thread
//               per query row, online softmax in base 2 with fp32 statistics,
//               lazy rescaling of O in tensor memory, and the epilogue.
// Work items, multi-head items for sequences of at most 128 / 64 tokens, masks
// and bounded waits as in the head_dim-64 kernel.
//
// Tensor memory (512 columns): S0/P0 [0,128) S1/P1 [128,256) O0 [256,384)
// O1 [384,512).
#include <cudaTypedefs.h>

#include "pe_kernels.cuh"
#include "pe_sm103.cuh"

namespace pe {

namespace {

using namespace sm103;

constexpr int kRows = 128;                         // query rows per tile = keys per block
constexpr int kD = 128;                            // head_dim
constexpr int kStages = 2;                         // K/V ring depth
constexpr int kIssueWarps = 3;
constexpr int kThreads = 384;
constexpr uint32_t kRegsLaunch = 168;
constexpr uint32_t kRegsLow = 56, kRegsHigh = 224;
static_assert(128 * (kRegsLow + 2 * kRegsHigh) <= kThreads * kRegsLaunch,
              "register split exceeds the launch allocation");
constexpr uint32_t kHalfColBytes = kRows * 64 * 2;   // one 64-column box of 128 rows: 16 KiB
constexpr uint32_t kTileBytes = 2 * kHalfColBytes;   // 32 KiB
constexpr uint32_t kHalfRowBytes = kHalfColBytes / 2;  // 64 rows of one 64-column box
constexpr int kPairRows = 2 * kRows;
// Output staging: 32 rows x 64 columns of a softmax warp (4 KiB, 128-byte
// swizzled), one 64-column half of its rows at a time, written by TMA.
constexpr uint32_t kStageWarpBytes = 32 * 64 * 2;

__host__ __device__ constexpr uint32_t col_s(int t) { return 128u * t; }   // P over its first 64
__host__ __device__ constexpr uint32_t col_o(int t) { return 256u + 128u * t; }
constexpr uint32_t kTmemCols = 512;

// kTailPair: the last query tiles of two heads of a longer sequence with an
// odd number of 128-row blocks; tile t runs head + t against its own head's
// key blocks, which alternate with the other tile's in the K/V ring.
enum : int32_t { kOneHead = 0, kHeadPerTile = 1, kTwoHeadsPerTile = 2, kTailPair = 3 };
struct Item {
  int32_t seq, head, pair;
  int32_t multi;
};

struct alignas(1024) Smem {
  __nv_bfloat16 q[2][kRows * kD];
  __nv_bfloat16 k[kStages][kRows * kD];
  __nv_bfloat16 v[kStages][kRows * kD];
  alignas(1024) uint8_t ostage[8][kStageWarpBytes];
  uint64_t item_full[2], item_empty[2];
  uint64_t q_full, q_empty;
  uint64_t k_full[kStages], v_full[kStages], k_empty[kStages], v_empty[kStages];
  uint64_t s_full[2], p_full[2], pv_done[2], o_full[2];
  uint64_t drain[kIssueWarps];
  Item items[2];
  uint32_t tmem_base;
  WaitGuard guard;
};

static_assert(sizeof(Smem) + 1024 <= 227 * 1024, "shared memory exceeds the per-CTA limit");

struct FwdParams {
  const int32_t* cu;
  int32_t B, H;
  int32_t pair_heads_rows;
  int32_t quad_heads_rows;
  int32_t pair_odd_tails;
  float scale_log2;
  __nv_bfloat16* out;
  float* lse;
  int64_t lse_stride;
  TilePlan plan;
  DeviceStatus* status;
  uint64_t wait_limit_ns;
};

enum WaitSite { kSiteProducer = 41, kSiteMma = 42, kSiteSoftmax = 43 };

__device__ __forceinline__ int item_tiles(const FwdParams& p, const Item& it, int32_t len) {
  if (it.multi == kHeadPerTile || it.multi == kTailPair) return 2;
  if (it.multi == kTwoHeadsPerTile) return p.H - it.head > 2 ? 2 : 1;
  return len - it.pair * kPairRows > kRows ? 2 : 1;
}

// Key blocks of an item: the whole sequence, or for multi-head items one block
// per tile (block t holds tile t's heads and serves only tile t), or for a
// kTailPair item both heads' blocks alternating (block j: head + (j & 1), keys
// 128 * (j / 2) ..).
__device__ __forceinline__ int32_t item_blocks(const Item& it, int32_t len, int ntiles) {
  if (it.multi == kTailPair) return 2 * ((len + kRows - 1) / kRows);
  return it.multi ? ntiles : (len + kRows - 1) / kRows;
}

// Blocks first(t), first(t) + step, ..., last(t) of the item serve tile t.
__device__ __forceinline__ bool tile_uses(const Item& it, int t, int32_t j) {
  if (it.multi == kTailPair) return (j & 1) == t;
  return it.multi ? j == t : true;
}

__device__ __forceinline__ void decode_item(const FwdParams& p, int32_t t, Item& it) {
  int32_t seq, local;
  plan_decode(p.plan.order, p.plan.tile_end, p.B, t, seq, local);
  const int32_t len = __ldg(p.cu + seq + 1) - __ldg(p.cu + seq);
  it.seq = seq;
  it.pair = 0;
  if (len <= p.quad_heads_rows) {
    it.head = 4 * local;
    it.multi = kTwoHeadsPerTile;
    return;
  }
  if (len <= p.pair_heads_rows) {
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

__device__ __forceinline__ int32_t packed_head(const FwdParams& p, const Item& it, int t, int hh) {
  const int32_t h = it.head + 2 * t + hh;
  return h < p.H ? h : it.head + 2 * t;
}

// A 128 x 128 tile as two 64-column boxes (each 128 rows, 16 KiB), or for a
// two-heads-per-tile item four 64-row boxes: rows 0-63 head a, 64-127 head b.
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* map,
                                          const CUtensorMap* map64, uint32_t bar, bool packed,
                                          int32_t x, int32_t y, int32_t xa, int32_t xb) {
  if (packed) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      tma_load_2d(dst + c * kHalfColBytes, map64, bar, xa + 64 * c, y);
      tma_load_2d(dst + c * kHalfColBytes + kHalfRowBytes, map64, bar, xb + 64 * c, y);
    }
  } else {
#pragma unroll
    for (int c = 0; c < 2; ++c) tma_load_2d(dst + c * kHalfColBytes, map, bar, x + 64 * c, y);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
fwd_sm103_d128_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_q64,
                      const __grid_constant__ CUtensorMap tm_k64,
                      const __grid_constant__ CUtensorMap tm_v64,
                      const __grid_constant__ CUtensorMap tm_o, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  Smem& S = *reinterpret_cast<Smem*>(smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile WaitGuard* abort_flag = &S.guard;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&S.item_full[i]), 1);
      mbar_init(smem_u32(&S.item_empty[i]), kIssueWarps + 8);
      mbar_init(smem_u32(&S.s_full[i]), 1);
      mbar_init(smem_u32(&S.pv_done[i]), 1);
      mbar_init(smem_u32(&S.p_full[i]), 4);
      mbar_init(smem_u32(&S.o_full[i]), 1);
    }
    mbar_init(smem_u32(&S.q_full), 1);
    mbar_init(smem_u32(&S.q_empty), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&S.k_full[s]), 1);
      mbar_init(smem_u32(&S.v_full[s]), 1);
      mbar_init(smem_u32(&S.k_empty[s]), 1);
      mbar_init(smem_u32(&S.v_empty[s]), 2);
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

  if (warp < 4) {
    regs_release<kRegsLow>();
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        uint32_t kv_no = 0;
        int pending_q = -1;
        int pending_k[kStages], pending_v[kStages];
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
          const int32_t nkv = item_blocks(it, len, ntiles);
          const int32_t x = it.head * kD;
          const bool packed = it.multi == kTwoHeadsPerTile;
          if (!mbar_wait(smem_u32(&S.q_empty), (item_no & 1) ^ 1, abort_flag, p.status,
                         kSiteProducer)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(smem_u32(&S.q_full), ntiles * kTileBytes);
          const bool tail = it.multi == kTailPair;
          for (int tt = 0; tt < ntiles; ++tt)
            load_tile(smem_u32(S.q[tt]), &tm_q, &tm_q64, smem_u32(&S.q_full), packed,
                      it.multi ? x + tt * kD : x,
                      tail ? start + r0 : (it.multi ? start : start + r0 + tt * kRows),
                      packed_head(p, it, tt, 0) * kD, packed_head(p, it, tt, 1) * kD);
          pending_q = item_no & 1;
          for (int32_t j = 0; j < nkv; ++j, ++kv_no) {
            const int s = kv_no % kStages;
            const uint32_t ph = (kv_no / kStages) & 1;
            const int32_t kx = tail ? x + (j & 1) * kD : (it.multi ? x + j * kD : x);
            const int32_t ky = tail ? start + (j >> 1) * kRows
                                    : (it.multi ? start : start + j * kRows);
            const int32_t xa = packed_head(p, it, j, 0) * kD, xb = packed_head(p, it, j, 1) * kD;
            if (!mbar_wait(smem_u32(&S.k_empty[s]), ph ^ 1, abort_flag, p.status, kSiteProducer)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(smem_u32(&S.k_full[s]), kTileBytes);
            load_tile(smem_u32(S.k[s]), &tm_k, &tm_k64, smem_u32(&S.k_full[s]), packed, kx, ky,
                      xa, xb);
            pending_k[s] = (int)ph;
            if (!mbar_wait(smem_u32(&S.v_empty[s]), ph ^ 1, abort_flag, p.status, kSiteProducer)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(smem_u32(&S.v_full[s]), kTileBytes);
            load_tile(smem_u32(S.v[s]), &tm_v, &tm_v64, smem_u32(&S.v_full[s]), packed, kx, ky,
                      xa, xb);
            pending_v[s] = (int)ph;
          }
        }
        if (!ok) {
          if (pending_q >= 0) mbar_drain_wait(smem_u32(&S.q_full), (uint32_t)pending_q);
          for (int s = 0; s < kStages; ++s) {
            if (pending_k[s] >= 0) mbar_drain_wait(smem_u32(&S.k_full[s]), (uint32_t)pending_k[s]);
            if (pending_v[s] >= 0) mbar_drain_wait(smem_u32(&S.v_full[s]), (uint32_t)pending_v[s]);
          }
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ QK issuer (whole warp)
      // The scores of a tile's next block overwrite the columns that hold this
      // block's P: they wait until P_t V of this block has completed.
      constexpr uint32_t idesc_qk = idesc_bf16(kRows, kRows, false, false);
      uint32_t kv_no = 0;
      uint32_t n_qk[2] = {0, 0};
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
        const int ntiles = item_tiles(p, it, len);
        const int32_t nkv = item_blocks(it, len, ntiles);
        if (!warp_wait(smem_u32(&S.q_full), item_no & 1, abort_flag, p.status, kSiteMma)) break;
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
            if (!tile_uses(it, t, j)) continue;
            if (n_qk[t] > 0 && !warp_wait(smem_u32(&S.pv_done[t]), (n_qk[t] - 1) & 1, abort_flag,
                                          p.status, kSiteMma)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t q_addr = smem_u32(S.q[t]);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kHalfColBytes + (kk & 3) * 32;
              mma_ss_warp(tmem + col_s(t), smem_desc_sw128(q_addr + off, 16, 1024),
                          smem_desc_sw128(k_addr + off, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
            }
            tc_commit_warp(smem_u32(&S.s_full[t]));
            ++n_qk[t];
          }
          if (!ok) break;
          tc_commit_warp(smem_u32(&S.k_empty[s]));
        }
        kv_no += nkv;
        if (ok) tc_commit_warp(smem_u32(&S.q_empty));
      }
      tc_commit_warp(smem_u32(&S.drain[0]));
      mbar_drain_wait(smem_u32(&S.drain[0]), 0);
    } else if (warp == 2 || warp == 3) {
      // ------------------------------------------------------------ PV issuers (whole warps)
      const int t = warp - 2;
      constexpr uint32_t idesc_pv = idesc_bf16(kRows, 64, false, true);
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
        const int ntiles = item_tiles(p, it, len);
        const int32_t nkv = item_blocks(it, len, ntiles);
        const bool tail = it.multi == kTailPair;
        const int32_t first = it.multi ? t : 0;
        const int32_t last = tail ? nkv - 2 + t : (it.multi ? t : nkv - 1);
        for (int32_t j = 0; j < nkv; ++j) {
          const uint32_t c = kv_no + j;
          const int s = c % kStages;
          if (!warp_wait(smem_u32(&S.v_full[s]), (c / kStages) & 1, abort_flag, p.status,
                         kSiteMma)) {
            ok = false;
            break;
          }
          if (t >= ntiles || !tile_uses(it, t, j)) {
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
#pragma unroll
            for (int nh = 0; nh < 2; ++nh)
              mma_ts_warp(tmem + col_o(t) + 64 * nh, tmem + col_s(t) + kk * 8,
                          smem_desc_sw128(v_addr + nh * kHalfColBytes + kk * 16 * 128, 16, 1024),
                          idesc_pv, (j > first || kk > 0) ? 1u : 0u);
          tc_commit_warp(smem_u32(&S.pv_done[t]));
          if (j == last) tc_commit_warp(smem_u32(&S.o_full[t]));
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
    const int t = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    uint32_t s_cnt = 0, o_cnt = 0;
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
      const int ntiles = item_tiles(p, it, len);
      if (t >= ntiles) continue;
      const bool packed = it.multi == kTwoHeadsPerTile;
      const bool tail = it.multi == kTailPair;
      const int32_t r0 = tail ? it.pair * kPairRows : (it.multi ? 0 : it.pair * kPairRows + t * kRows);
      const int32_t head = packed ? it.head + 2 * t + (quarter >> 1)
                                  : (it.multi ? it.head + t : it.head);
      const int32_t pos = packed ? (row & 63) : r0 + row;
      const int32_t coff = packed ? (quarter >> 1) * 64 : 0;
      const int32_t nkv = item_blocks(it, len, ntiles);
      const int32_t first = it.multi ? t : 0;
      const int32_t last = tail ? nkv - 2 + t : (it.multi ? t : nkv - 1);
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int32_t j = first; j <= last; j += tail ? 2 : 1) {
        const bool first_blk = j == first;
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
        const int32_t kb = tail ? (j >> 1) * kRows : (it.multi ? 0 : j * kRows);
        const int32_t kv_valid = len - kb;
        if (kv_valid < kRows) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (32 * c + e < coff || 32 * c + e >= coff + kv_valid) sr[c][e] = 0xff800000u;
        }
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
        const bool grow = m_blk > m + 8.f;
        const float m_new = grow ? m_blk : m;
        const float alpha = grow ? ex2(m - m_new) : 1.f;
        const uint64_t c2 = f2(scale_log2, scale_log2), nm2 = f2(-m_new, -m_new);
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
        // P over the first 64 score columns: the scores are in registers, and
        // the previous P V (which read the old P there) completed before these
        // scores were computed.
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_st16(lane_base + col_s(t) + 16 * c, pk[c]);
        // O holds P(j-1) V(j-1) (complete, for the same reason): rescale it
        // when some row's maximum moved.
        if (!first_blk && __any_sync(0xffffffffu, grow)) {
#pragma unroll
          for (int h = 0; h < 4; ++h) {
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
      // A warp's 32 rows are 32 consecutive tokens of one head: when all are
      // real, each 64-column half goes through the warp's 4 KiB stage to one
      // TMA store; the partial warp at a sequence's end stores its rows itself.
      const bool store = pos < len && head < p.H;
      const bool full = head < p.H && len - (pos - lane) >= 32;   // warp-uniform
      const int64_t tok = static_cast<int64_t>(start) + pos;
      const float inv = 1.f / l;
      uint8_t* stage = S.ostage[warp - 4];
      uint4* dst = reinterpret_cast<uint4*>(p.out + (tok * p.H + head) * kD);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t o[2][32];
        tmem_ld32(lane_base + col_o(t) + 64 * c, o[0]);
        tmem_ld32(lane_base + col_o(t) + 64 * c + 32, o[1]);
        tmem_wait_ld(o[0]);
        tmem_wait_ld(o[1]);
        if (full) {
          if (lane == 0) bulk_wait_read();   // the previous half has left the stage
          __syncwarp();
        }
        if (full || store) {
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const uint32_t* src = o[g >> 2] + (g & 3) * 8;
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(src[0]) * inv, __uint_as_float(src[1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(src[2]) * inv, __uint_as_float(src[3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(src[4]) * inv, __uint_as_float(src[5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(src[6]) * inv, __uint_as_float(src[7]) * inv);
            if (full)
              *reinterpret_cast<uint4*>(stage + lane * 128 + ((g ^ (lane & 7)) << 4)) = w;
            else
              dst[8 * c + g] = w;
          }
        }
        if (full) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tm_o, smem_u32(stage), head * kD + 64 * c, start + (pos - lane));
            bulk_commit();
          }
        }
      }
      if (store && p.lse) p.lse[static_cast<int64_t>(head) * p.lse_stride + tok] =
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
PFN_cuTensorMapEncodeTiled_v12000 g_encode_d128 = nullptr;

pe_status get_encoder_d128() {
  if (g_encode_d128) return PE_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult qres;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &qres) != cudaSuccess ||
      qres != cudaDriverEntryPointSuccess || !fn)
    return PE_ERR_CUDA;
  g_encode_d128 = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return PE_OK;
}

// [N, H*128] bf16 rows; boxes of box_rows rows x 64 columns (half a head),
// 128-byte swizzle.
pe_status make_map_d128(CUtensorMap* map, const void* base, int64_t N, int32_t H,
                        uint32_t box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(H) * kD, static_cast<cuuint64_t>(N)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * kD * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t elem_strides[2] = {1, 1};
  CUresult r = g_encode_d128(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
                             dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PE_OK : PE_ERR_CUDA;
}

}  // namespace

int sm103_d128_fwd_rows_per_item() { return kPairRows; }
int sm103_d128_fwd_pair_heads_rows() { return kRows; }
int sm103_d128_fwd_quad_heads_rows() { return kRows / 2; }
int sm103_d128_fwd_pair_odd_tails() { return 1; }

pe_status fwd_sm103_d128(const void* q, const void* k, const void* v, const int32_t* cu,
                         int32_t B, int32_t H, int64_t N, float scale, void* out, float* lse,
                         TilePlan plan, DeviceStatus* status, cudaStream_t stream) {
  PE_TRY(get_encoder_d128());
  CUtensorMap mq, mk, mv, mq64, mk64, mv64, mo;
  PE_TRY(make_map_d128(&mo, out, N, H, 32));
  PE_TRY(make_map_d128(&mq, q, N, H, kRows));
  PE_TRY(make_map_d128(&mk, k, N, H, kRows));
  PE_TRY(make_map_d128(&mv, v, N, H, kRows));
  PE_TRY(make_map_d128(&mq64, q, N, H, 64));
  PE_TRY(make_map_d128(&mk64, k, N, H, 64));
  PE_TRY(make_map_d128(&mv64, v, N, H, 64));
  const size_t smem = sizeof(Smem) + 1024;
  PE_CUDA_TRY(cudaFuncSetAttribute(fwd_sm103_d128_kernel,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(smem)));
  cudaFuncAttributes attr;
  PE_CUDA_TRY(cudaFuncGetAttributes(&attr, fwd_sm103_d128_kernel));
  if (static_cast<uint32_t>(attr.numRegs) * kThreads < 128u * (kRegsLow + 2 * kRegsHigh))
    return PE_ERR_UNSUPPORTED;
  FwdParams prm;
  prm.cu = cu;
  prm.B = B;
  prm.H = H;
  prm.pair_heads_rows = sm103_d128_fwd_pair_heads_rows();
  prm.quad_heads_rows = sm103_d128_fwd_quad_heads_rows();
  prm.pair_odd_tails = sm103_d128_fwd_pair_odd_tails();
  prm.scale_log2 = scale * kLog2e;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.lse = lse;
  prm.lse_stride = N;
  prm.plan = plan;
  prm.status = status;
  prm.wait_limit_ns = wait_limit_ns();
  PE_TRY(launch_after_previous(fwd_sm103_d128_kernel, dim3(device_sm_count()), dim3(kThreads),
                               smem, stream, mq, mk, mv, mq64, mk64, mv64, mo, prm));
  PE_CUDA_TRY(cudaGetLastError());
  return PE_OK;
}

}  // namespace pe
