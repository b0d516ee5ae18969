// Packed attention forward on the sm_103a tensor cores for fp32 inputs and
// outputs, head_dim 64 (page "Source code for gigl.nn.packed_attention":
// every sequence attends only to itself within its cu_seqlens bounds; the
// memory-efficient kernel the page calls runs in fp32 "which inference needs
// for accuracy", function _varlen_attention).
//
// fp32 accuracy from bf16 tensor-core products: every fp32 operand x is split
// into two bf16 parts, hi = bf16(x) and lo = bf16(x - hi) (round to nearest
// even both times), so that |x - hi - lo| <= 2^-18 |x|, and each product is
// taken as hi*hi + hi*lo + lo*hi (the dropped lo*lo is below 2^-18 of it):
//   S = Qhi Khi^T + Qhi Klo^T + Qlo Khi^T,   O += Phi Vhi + Phi Vlo + Plo Vhi,
// all accumulated in fp32 in tensor memory. A score then carries an error of
// at most ~3 * 2^-18 * scale * sum_c |q_c k_c| and an output row one of the
// same relative size, well inside the fp32 bar of 1e-4 for inputs of unit
// scale; the softmax statistics stay in fp32 throughout.
//
// Design (one persistent CTA per SM, 16 warps), following the bf16 kernel:
//   warp 0       producer: claims work items from the longest-first plan and
//                publishes them to a two-slot ring; streams the raw fp32 Q
//                tiles and K/V blocks (128 rows x 64, no swizzle) with TMA.
//   warps 12-15  split: turn each landed fp32 tile, in place, into its bf16 hi
//                and lo operands in the 128-byte-swizzled layout the MMAs
//                read. The raw rows 8g..8g+7 (2 KiB) become the hi atom g (the
//                first KiB) and the lo atom g (the second), so each warp
//                converts whole 8-row groups on its own: the hi and lo operands
//                are interleaved atom by atom, 2 KiB apart.
//   warp 1       issues S = Q_t K_j^T for both query tiles in turn into ONE
//                shared score buffer (tensor memory holds 512 columns: S, and
//                per tile P hi, P lo and O), as soon as the other tile's
//                softmax has read the previous scores.
//   warps 2, 3   issue O_t += P_t V_j for tile 0 and tile 1.
//   warps 4-7    softmax of query tile 0; warps 8-11 of query tile 1: one
//   and 8-11     thread per query row, online softmax in base 2 with fp32
//                statistics, P split into hi and lo bf16 halves in tensor
//                memory, O rescaled in tensor memory when the row maximum grows
//                by more than 2^8, and the epilogue (normalise, store, lse).
// A work item is (sequence, head, pair of 128-row query tiles); sequences of
// at most 128 tokens run one head per tile, sequences of at most 64 tokens two
// heads per tile (rows 0-63 and 64-127), as in the bf16 kernel. Keys past the
// sequence end are masked to -inf; query rows past it are computed but never
// stored. TMA zero-fills rows beyond the packed buffer.
//
// Tensor memory (512 columns): S [0,128); tile t: P hi [128+192t, +64),
// P lo [192+192t, +64), O [256+192t, +64).
//
// Every wait is bounded (pe_set_wait_limit_ns): the CTA then records
// PE_ERR_DEVICE_TIMEOUT, drains its own copies and MMAs, frees tensor memory
// and exits. No two warps share a named barrier, so no warp can be left
// waiting for one that gave up.
#include <cudaTypedefs.h>

#include "pe_kernels.cuh"
#include "pe_sm103.cuh"

namespace pe {

namespace {

using namespace sm103;

constexpr int kRows = 128;                         // query rows per tile = keys per block
constexpr int kD = 64;                             // head_dim
constexpr int kStages = 2;                         // K/V ring depth
constexpr int kIssueWarps = 3;                     // QK issuer + one PV issuer per tile
constexpr int kSplitWarps = 4;
constexpr int kThreads = 512;
// Registers per thread: 128 at launch (one CTA of 512 threads per SM); the
// producer/issuer warpgroup drops to kRegsLow, the split warpgroup to
// kRegsSplit and the two softmax warpgroups rise to kRegsHigh.
constexpr uint32_t kRegsLaunch = 65536 / kThreads;
constexpr uint32_t kRegsLow = 56, kRegsSplit = 56, kRegsHigh = 200;
static_assert(128 * (kRegsLow + kRegsSplit + 2 * kRegsHigh) <= kThreads * kRegsLaunch,
              "register split exceeds the launch allocation");
constexpr uint32_t kRawTileBytes = kRows * kD * 4;   // 32 KiB of fp32
constexpr uint32_t kRawHalfBytes = kRawTileBytes / 2;  // 64 rows
// Split operands: 8-row atoms of 1 KiB, hi atom g at 2 KiB * g, lo atom g 1 KiB
// after it, so consecutive atoms of one operand are kAtomStride apart.
constexpr uint32_t kLoOffset = 1024;
constexpr uint32_t kAtomStride = 2048;
constexpr int kPairRows = 2 * kRows;                 // query rows per work item

// Tensor-memory columns.
constexpr uint32_t kColS = 0;
__host__ __device__ constexpr uint32_t col_phi(int t) { return 128u + 192u * t; }
__host__ __device__ constexpr uint32_t col_plo(int t) { return 192u + 192u * t; }
__host__ __device__ constexpr uint32_t col_o(int t) { return 256u + 192u * t; }
constexpr uint32_t kTmemCols = 512;

enum : int32_t { kOneHead = 0, kHeadPerTile = 1, kTwoHeadsPerTile = 2 };
struct Item {
  int32_t seq, head, pair;
  int32_t multi;
};

struct alignas(1024) Smem {
  // Raw fp32 tiles; after the split each holds its hi and lo bf16 operands,
  // atom by atom.
  float q[2][kRows * kD];
  float k[kStages][kRows * kD];
  float v[kStages][kRows * kD];
  uint64_t item_full[2], item_empty[2];
  uint64_t q_raw, q_full, q_empty;
  uint64_t k_raw[kStages], v_raw[kStages];
  uint64_t k_full[kStages], v_full[kStages], k_empty[kStages], v_empty[kStages];
  uint64_t s_full[2], s_free, p_full[2], pv_done[2], o_full[2];
  uint64_t drain[kIssueWarps];
  Item items[2];
  uint32_t tmem_base;
  WaitGuard guard;
};

struct FwdParams {
  const int32_t* cu;
  int32_t B, H;
  int32_t pair_heads_rows;  // sequences up to this long run a head per tile
  int32_t quad_heads_rows;  // ... and up to this long two heads per tile
  float scale_log2;
  float* out;
  float* lse;
  int64_t lse_stride;
  TilePlan plan;
  DeviceStatus* status;
  uint64_t wait_limit_ns;
};

enum WaitSite { kSiteProducer = 31, kSiteMma = 32, kSiteSoftmax = 33, kSiteSplit = 34 };

__device__ __forceinline__ int item_tiles(const FwdParams& p, const Item& it, int32_t len) {
  if (it.multi == kHeadPerTile) return 2;
  if (it.multi == kTwoHeadsPerTile) return p.H - it.head > 2 ? 2 : 1;
  return len - it.pair * kPairRows > kRows ? 2 : 1;
}

// Key blocks of an item: the whole sequence for ordinary items; for
// multi-head items block t holds tile t's heads and serves only tile t.
__device__ __forceinline__ int32_t item_blocks(const Item& it, int32_t len, int ntiles) {
  return it.multi ? ntiles : (len + kRows - 1) / kRows;
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
  it.head = local / npairs;
  it.pair = local - it.head * npairs;
  it.multi = kOneHead;
}

__device__ __forceinline__ int32_t packed_head(const FwdParams& p, const Item& it, int t, int hh) {
  const int32_t h = it.head + 2 * t + hh;
  return h < p.H ? h : it.head + 2 * t;
}

// Splits one landed fp32 tile (128 rows x 64, row-major) in place. The 8-row
// group g (raw bytes [2 KiB g, 2 KiB (g+1))) becomes the hi atom g in its first
// KiB and the lo atom g in its second, each 128-byte swizzled: the 16-byte
// chunk m of atom row r sits at r * 128 + ((m ^ r) * 16). Warp w of the four
// split warps converts groups w, w + 4, w + 8 and w + 12, two at a time; lane
// l takes the float4s l, l + 32, l + 64 and l + 96 of a group (row f / 16,
// columns 4 (f % 16) .. +3 for float4 f), i.e. half of a bf16 chunk of each.
__device__ __forceinline__ void split_tile(float* tile, int w, int lane) {
  uint8_t* base = reinterpret_cast<uint8_t*>(tile);
#pragma unroll
  for (int gi = 0; gi < 4; gi += 2) {
    float4 x[2][4];
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      const float4* grp = reinterpret_cast<const float4*>(base + kAtomStride * (w + 4 * (gi + a)));
#pragma unroll
      for (int k = 0; k < 4; ++k) x[a][k] = grp[lane + 32 * k];
    }
    __syncwarp();  // every raw value of the two groups is read before any is overwritten
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      uint8_t* grp = base + kAtomStride * (w + 4 * (gi + a));
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int f = lane + 32 * k, r = f >> 4, col4 = f & 15;
        const uint32_t h0 = pack_bf16x2(x[a][k].x, x[a][k].y);
        const uint32_t h1 = pack_bf16x2(x[a][k].z, x[a][k].w);
        const uint32_t l0 = pack_bf16x2(x[a][k].x - __uint_as_float(h0 << 16),
                                        x[a][k].y - __uint_as_float(h0 & 0xffff0000u));
        const uint32_t l1 = pack_bf16x2(x[a][k].z - __uint_as_float(h1 << 16),
                                        x[a][k].w - __uint_as_float(h1 & 0xffff0000u));
        const uint32_t off = r * 128 + (((col4 >> 1) ^ r) << 4) + 8 * (col4 & 1);
        *reinterpret_cast<uint2*>(grp + off) = make_uint2(h0, h1);
        *reinterpret_cast<uint2*>(grp + kLoOffset + off) = make_uint2(l0, l1);
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
fwd_sm103_f32_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_q64,
                     const __grid_constant__ CUtensorMap tm_k64,
                     const __grid_constant__ CUtensorMap tm_v64, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  Smem& S = *reinterpret_cast<Smem*>(smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile WaitGuard* abort_flag = &S.guard;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&S.item_full[i]), 1);
      mbar_init(smem_u32(&S.item_empty[i]), kIssueWarps + 8 + kSplitWarps);
      mbar_init(smem_u32(&S.s_full[i]), 1);
      mbar_init(smem_u32(&S.pv_done[i]), 1);
      mbar_init(smem_u32(&S.p_full[i]), 4);
      mbar_init(smem_u32(&S.o_full[i]), 1);
    }
    mbar_init(smem_u32(&S.s_free), 4);              // the softmax warps of the tile that read S
    mbar_init(smem_u32(&S.q_raw), 1);
    mbar_init(smem_u32(&S.q_full), kSplitWarps);
    mbar_init(smem_u32(&S.q_empty), 1);             // the QK issuer, after an item's last QK
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&S.k_raw[s]), 1);
      mbar_init(smem_u32(&S.v_raw[s]), 1);
      mbar_init(smem_u32(&S.k_full[s]), kSplitWarps);
      mbar_init(smem_u32(&S.v_full[s]), kSplitWarps);
      mbar_init(smem_u32(&S.k_empty[s]), 1);        // the QK issuer, after both tiles' QK
      mbar_init(smem_u32(&S.v_empty[s]), 2);        // each PV issuer, once per block
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
          mbar_arrive_expect_tx(smem_u32(&S.q_raw), ntiles * kRawTileBytes);
          for (int tt = 0; tt < ntiles; ++tt) {
            if (packed) {
              for (int hh = 0; hh < 2; ++hh)
                tma_load_2d(smem_u32(S.q[tt]) + hh * kRawHalfBytes, &tm_q64, smem_u32(&S.q_raw),
                            packed_head(p, it, tt, hh) * kD, start);
            } else {
              tma_load_2d(smem_u32(S.q[tt]), &tm_q, smem_u32(&S.q_raw),
                          it.multi ? x + tt * kD : x, it.multi ? start : start + r0 + tt * kRows);
            }
          }
          pending_q = item_no & 1;
          for (int32_t j = 0; j < nkv; ++j, ++kv_no) {
            const int s = kv_no % kStages;
            const uint32_t ph = (kv_no / kStages) & 1;
            const int32_t kx = it.multi ? x + j * kD : x;
            const int32_t ky = it.multi ? start : start + j * kRows;
            if (!mbar_wait(smem_u32(&S.k_empty[s]), ph ^ 1, abort_flag, p.status, kSiteProducer)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(smem_u32(&S.k_raw[s]), kRawTileBytes);
            if (packed) {
              for (int hh = 0; hh < 2; ++hh)
                tma_load_2d(smem_u32(S.k[s]) + hh * kRawHalfBytes, &tm_k64, smem_u32(&S.k_raw[s]),
                            packed_head(p, it, j, hh) * kD, start);
            } else {
              tma_load_2d(smem_u32(S.k[s]), &tm_k, smem_u32(&S.k_raw[s]), kx, ky);
            }
            pending_k[s] = (int)ph;
            if (!mbar_wait(smem_u32(&S.v_empty[s]), ph ^ 1, abort_flag, p.status, kSiteProducer)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(smem_u32(&S.v_raw[s]), kRawTileBytes);
            if (packed) {
              for (int hh = 0; hh < 2; ++hh)
                tma_load_2d(smem_u32(S.v[s]) + hh * kRawHalfBytes, &tm_v64, smem_u32(&S.v_raw[s]),
                            packed_head(p, it, j, hh) * kD, start);
            } else {
              tma_load_2d(smem_u32(S.v[s]), &tm_v, smem_u32(&S.v_raw[s]), kx, ky);
            }
            pending_v[s] = (int)ph;
          }
        }
        if (!ok) {
          // Let every copy this thread started land before the CTA exits.
          if (pending_q >= 0) mbar_drain_wait(smem_u32(&S.q_raw), (uint32_t)pending_q);
          for (int s = 0; s < kStages; ++s) {
            if (pending_k[s] >= 0) mbar_drain_wait(smem_u32(&S.k_raw[s]), (uint32_t)pending_k[s]);
            if (pending_v[s] >= 0) mbar_drain_wait(smem_u32(&S.v_raw[s]), (uint32_t)pending_v[s]);
          }
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ QK issuer (whole warp)
      // One score buffer serves both tiles in turn: QK number n waits until the
      // scores of QK number n - 1 have been read by their tile's softmax.
      constexpr uint32_t idesc_qk = idesc_bf16(kRows, kRows, false, false);
      uint32_t kv_no = 0, n_s = 0;
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
          const uint32_t khi = smem_u32(S.k[s]), klo = khi + kLoOffset;
          for (int t = 0; t < ntiles; ++t) {
            if (it.multi && j != t) continue;   // the other tile's heads
            if (n_s > 0 && !warp_wait(smem_u32(&S.s_free), (n_s - 1) & 1, abort_flag, p.status,
                                      kSiteMma)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t qhi = smem_u32(S.q[t]), qlo = qhi + kLoOffset;
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              mma_ss_warp(tmem + kColS, smem_desc_sw128(qhi + kk * 32, 16, kAtomStride),
                          smem_desc_sw128(khi + kk * 32, 16, kAtomStride), idesc_qk,
                          kk > 0 ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              mma_ss_warp(tmem + kColS, smem_desc_sw128(qhi + kk * 32, 16, kAtomStride),
                          smem_desc_sw128(klo + kk * 32, 16, kAtomStride), idesc_qk, 1u);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              mma_ss_warp(tmem + kColS, smem_desc_sw128(qlo + kk * 32, 16, kAtomStride),
                          smem_desc_sw128(khi + kk * 32, 16, kAtomStride), idesc_qk, 1u);
            tc_commit_warp(smem_u32(&S.s_full[t]));
            ++n_s;
          }
          if (!ok) break;
          tc_commit_warp(smem_u32(&S.k_empty[s]));  // K_j no longer needed by either tile
        }
        kv_no += nkv;
        if (ok) tc_commit_warp(smem_u32(&S.q_empty));
      }
      tc_commit_warp(smem_u32(&S.drain[0]));
      mbar_drain_wait(smem_u32(&S.drain[0]), 0);
    } else if (warp == 2 || warp == 3) {
      // ------------------------------------------------------------ PV issuers (whole warps)
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
        const int ntiles = item_tiles(p, it, len);
        const int32_t nkv = item_blocks(it, len, ntiles);
        const int32_t first = it.multi ? t : 0, last = it.multi ? t : nkv - 1;
        for (int32_t j = 0; j < nkv; ++j) {
          const uint32_t c = kv_no + j;
          const int s = c % kStages;
          // Both PV warps take part in every V stage phase.
          if (!warp_wait(smem_u32(&S.v_full[s]), (c / kStages) & 1, abort_flag, p.status,
                         kSiteMma)) {
            ok = false;
            break;
          }
          if (t >= ntiles || j < first || j > last) {  // this tile does not read V_j
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&S.v_empty[s]));
            continue;
          }
          if (!warp_wait(smem_u32(&S.p_full[t]), n_pv & 1, abort_flag, p.status, kSiteMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // A K-step of 16 keys spans two 8-row atoms of each operand.
          const uint32_t vhi = smem_u32(S.v[s]), vlo = vhi + kLoOffset;
#pragma unroll
          for (int kk = 0; kk < kRows / 16; ++kk)
            mma_ts_warp(tmem + col_o(t), tmem + col_phi(t) + kk * 8,
                        smem_desc_sw128(vhi + kk * 2 * kAtomStride, 16, kAtomStride), idesc_pv,
                        (j > first || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < kRows / 16; ++kk)
            mma_ts_warp(tmem + col_o(t), tmem + col_phi(t) + kk * 8,
                        smem_desc_sw128(vlo + kk * 2 * kAtomStride, 16, kAtomStride), idesc_pv,
                        1u);
#pragma unroll
          for (int kk = 0; kk < kRows / 16; ++kk)
            mma_ts_warp(tmem + col_o(t), tmem + col_plo(t) + kk * 8,
                        smem_desc_sw128(vhi + kk * 2 * kAtomStride, 16, kAtomStride), idesc_pv,
                        1u);
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
  } else if (warp >= 12) {
    regs_release<kRegsSplit>();
    // -------------------------------------------------------------- split warps
    // Each warp converts its own atoms and arrives on its own: a wait that
    // gives up ends only this warp's loop.
    const int w = warp - 12;
    uint32_t kv_no = 0;
    bool ok = true;
    for (uint32_t item_no = 0; ok; ++item_no) {
      const int slot = item_no & 1;
      if (!warp_wait(smem_u32(&S.item_full[slot]), (item_no >> 1) & 1, abort_flag, p.status,
                     kSiteSplit))
        break;
      const Item it = S.items[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&S.item_empty[slot]));
      if (it.seq < 0) break;
      const int32_t len = __ldg(p.cu + it.seq + 1) - __ldg(p.cu + it.seq);
      const int ntiles = item_tiles(p, it, len);
      const int32_t nkv = item_blocks(it, len, ntiles);
      if (!warp_wait(smem_u32(&S.q_raw), item_no & 1, abort_flag, p.status, kSiteSplit)) break;
      for (int tt = 0; tt < ntiles; ++tt) split_tile(S.q[tt], w, lane);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&S.q_full));
      for (int32_t j = 0; j < nkv; ++j, ++kv_no) {
        const int s = kv_no % kStages;
        const uint32_t ph = (kv_no / kStages) & 1;
        if (!warp_wait(smem_u32(&S.k_raw[s]), ph, abort_flag, p.status, kSiteSplit)) {
          ok = false;
          break;
        }
        split_tile(S.k[s], w, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&S.k_full[s]));
        if (!warp_wait(smem_u32(&S.v_raw[s]), ph, abort_flag, p.status, kSiteSplit)) {
          ok = false;
          break;
        }
        split_tile(S.v[s], w, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&S.v_full[s]));
      }
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
      const int32_t r0 = it.multi ? 0 : it.pair * kPairRows + t * kRows;
      const int32_t head = packed ? it.head + 2 * t + (quarter >> 1)
                                  : (it.multi ? it.head + t : it.head);
      const int32_t pos = packed ? (row & 63) : r0 + row;
      const int32_t coff = packed ? (quarter >> 1) * 64 : 0;
      const int32_t nkv = item_blocks(it, len, ntiles);
      const int32_t first = it.multi ? t : 0, last = it.multi ? t : nkv - 1;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int32_t j = first; j <= last; ++j) {
        const bool first_blk = j == first;
        if (!warp_wait(smem_u32(&S.s_full[t]), s_cnt & 1, abort_flag, p.status, kSiteSoftmax)) {
          ok = false;
          break;
        }
        ++s_cnt;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + kColS + 32 * c, sr[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_wait_ld(sr[c]);
        // The scores are in registers: the other tile's QK may overwrite them.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&S.s_free));
        const int32_t kb = it.multi ? 0 : j * kRows;
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
            for (int w = 0; w < 4; ++w)
              mx[w] = max3(mx[w], __uint_as_float(sr[c][e + 2 * w]),
                           __uint_as_float(sr[c][e + 2 * w + 1]));
        const float m_blk = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * scale_log2;
        const bool grow = m_blk > m + 8.f;
        const float m_new = grow ? m_blk : m;
        const float alpha = grow ? ex2(m - m_new) : 1.f;
        const uint64_t c2 = f2(scale_log2, scale_log2), nm2 = f2(-m_new, -m_new);
        if (!first_blk) {
          // P_t(j-1) V must have finished before P_t is overwritten or O_t rescaled.
          if (!warp_wait(smem_u32(&S.pv_done[t]), (s_cnt - 2) & 1, abort_flag, p.status,
                         kSiteSoftmax)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        // Exponents 32 keys at a time, split into bf16 hi and lo pairs and
        // stored to tensor memory at once (each chunk's scores die as its
        // pairs are stored, which keeps the row within the register budget).
        uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint64_t x = ffma2(f2(__uint_as_float(sr[c][2 * e]),
                                        __uint_as_float(sr[c][2 * e + 1])), c2, nm2);
            float p0, p1;
            f2_split(x, p0, p1);
            p0 = ex2(p0);
            p1 = ex2(p1);
            acc[e & 3] = fadd2(acc[e & 3], f2(p0, p1));
            hi[e] = pack_bf16x2(p0, p1);
            lo[e] = pack_bf16x2(p0 - __uint_as_float(hi[e] << 16),
                                p1 - __uint_as_float(hi[e] & 0xffff0000u));
          }
          tmem_st16(lane_base + col_phi(t) + 16 * c, hi);
          tmem_st16(lane_base + col_plo(t) + 16 * c, lo);
        }
        float s0, s1, s2, s3, s4, s5, s6, s7;
        f2_split(acc[0], s0, s1);
        f2_split(acc[1], s2, s3);
        f2_split(acc[2], s4, s5);
        f2_split(acc[3], s6, s7);
        l = l * alpha + (((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7)));
        m = m_new;
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
      if (pos < len && head < p.H) {
        const int64_t tok = static_cast<int64_t>(start) + pos;
        const float inv = 1.f / l;
        float4* dst = reinterpret_cast<float4*>(p.out + (tok * p.H + head) * kD);
#pragma unroll
        for (int g = 0; g < 16; ++g) {
          const uint32_t* src = o[g >> 3] + (g & 7) * 4;
          dst[g] = make_float4(__uint_as_float(src[0]) * inv, __uint_as_float(src[1]) * inv,
                               __uint_as_float(src[2]) * inv, __uint_as_float(src[3]) * inv);
        }
        if (p.lse) p.lse[static_cast<int64_t>(head) * p.lse_stride + tok] =
            (m + __log2f(l)) * kLn2;
      }
    }
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
PFN_cuTensorMapEncodeTiled_v12000 g_encode_f32 = nullptr;

pe_status get_encoder_f32() {
  if (g_encode_f32) return PE_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult qres;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &qres) != cudaSuccess ||
      qres != cudaDriverEntryPointSuccess || !fn)
    return PE_ERR_CUDA;
  g_encode_f32 = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return PE_OK;
}

// [N, H*64] fp32 rows; boxes of box_rows rows x 64 columns (one head, 256
// bytes per row), no swizzle: the split warps read them row-major.
pe_status make_map_f32(CUtensorMap* map, const void* base, int64_t N, int32_t H,
                       uint32_t box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(H) * kD, static_cast<cuuint64_t>(N)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * kD * 4};
  cuuint32_t box[2] = {kD, box_rows};
  cuuint32_t elem_strides[2] = {1, 1};
  CUresult r = g_encode_f32(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base),
                            dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PE_OK : PE_ERR_CUDA;
}

}  // namespace

int sm103_f32_fwd_rows_per_item() { return kPairRows; }
int sm103_f32_fwd_pair_heads_rows() { return kRows; }
int sm103_f32_fwd_quad_heads_rows() { return kRows / 2; }

pe_status fwd_sm103_f32(const void* q, const void* k, const void* v, const int32_t* cu,
                        int32_t B, int32_t H, int64_t N, float scale, void* out, float* lse,
                        TilePlan plan, DeviceStatus* status, cudaStream_t stream) {
  PE_TRY(get_encoder_f32());
  CUtensorMap mq, mk, mv, mq64, mk64, mv64;
  PE_TRY(make_map_f32(&mq, q, N, H, kRows));
  PE_TRY(make_map_f32(&mk, k, N, H, kRows));
  PE_TRY(make_map_f32(&mv, v, N, H, kRows));
  PE_TRY(make_map_f32(&mq64, q, N, H, 64));
  PE_TRY(make_map_f32(&mk64, k, N, H, 64));
  PE_TRY(make_map_f32(&mv64, v, N, H, 64));
  const size_t smem = sizeof(Smem) + 1024;
  PE_CUDA_TRY(cudaFuncSetAttribute(fwd_sm103_f32_kernel,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(smem)));
  // The softmax warpgroups' register claim is served from what the CTA was
  // launched with; never launch a build whose count cannot serve it.
  cudaFuncAttributes attr;
  PE_CUDA_TRY(cudaFuncGetAttributes(&attr, fwd_sm103_f32_kernel));
  if (static_cast<uint32_t>(attr.numRegs) * kThreads <
      128u * (kRegsLow + kRegsSplit + 2 * kRegsHigh))
    return PE_ERR_UNSUPPORTED;
  FwdParams prm;
  prm.cu = cu;
  prm.B = B;
  prm.H = H;
  prm.pair_heads_rows = sm103_f32_fwd_pair_heads_rows();
  prm.quad_heads_rows = sm103_f32_fwd_quad_heads_rows();
  prm.scale_log2 = scale * kLog2e;
  prm.out = static_cast<float*>(out);
  prm.lse = lse;
  prm.lse_stride = N;
  prm.plan = plan;
  prm.status = status;
  prm.wait_limit_ns = wait_limit_ns();
  PE_TRY(launch_after_previous(fwd_sm103_f32_kernel, dim3(device_sm_count()), dim3(kThreads),
                               smem, stream, mq, mk, mv, mq64, mk64, mv64, prm));
  PE_CUDA_TRY(cudaGetLastError());
  return PE_OK;
}

}  // namespace pe
