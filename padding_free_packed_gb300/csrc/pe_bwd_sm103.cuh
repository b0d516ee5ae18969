// Packed attention backward on the sm_103a tensor cores, bf16, head_dim 64 or
// 128 (D): the gradients in q, k and v that the custom op
// gigl::varlen_attention_backward returns (page "Source code for
// gigl.nn.packed_attention"), recomputing P from the saved log-sum-exp.
// Deterministic (no floating-point atomics): two passes over 128-row blocks.
//
//   key pass   (one work item = 128 keys of one sequence and head; loops over
//              the sequence's 128-query blocks i):
//                S^T  = K Q_i^T,  dP^T = V dO_i^T             (M=128, N=128, K=64)
//                P^T  = exp2(S^T * scale*log2e - lse_q * log2e)
//                dS^T = P^T o (dP^T - Delta_q)                (per-query columns)
//                dV  += P^T dO_i,  dK += dS^T Q_i              (M=128, N=64, K=128)
//              dK is scaled once at the end.
//   query pass (one work item = 128 queries; loops over 128-key blocks j):
//                S = Q K_j^T, dP = dO V_j^T,  P = exp2(...lse_r), dS = P o (dP - Delta_r)
//                dQ += dS K_j,  scaled once at the end.
//
// One persistent CTA per SM, 16 warps:
//   warp 0       TMA producer: the item's two stationary tiles (K, V or Q, dO),
//                then a ring of streaming tile pairs (Q_i, dO_i or K_j, V_j);
//                in the key pass the warp also stages each block's lse and
//                Delta columns in shared memory.
//   warp 5       scheduler: claims work items from the longest-first plan and
//                decodes them into the two-slot item ring ahead of the
//                producer, so that the claim's atomic and the plan and
//                cu_seqlens reads are off the producer's per-item chain.
//   warps 1, 2   issue the two score-shaped products (warp 1 owns tensor memory).
//   warps 3, 4   issue the accumulations (warp 4 only in the key pass). A single
//                thread issues one tcgen05.mma per ~130 cycles, hence four issuers.
//   warps 8-15   elementwise step: warps 8-11 take columns 0-63, warps 12-15
//                columns 64-127; one thread per TMEM lane (tile row). A warp
//                loads its 64 columns of both products into registers and
//                releases them at once, so the next block's products run while
//                it computes P and dS; those are packed to bf16 and stored into
//                tensor memory once the previous block's accumulations have
//                read theirs. Then the epilogue (scale, store the rows inside
//                the sequence). Warps 0-7 hand registers to these (setmaxnreg).
// Tensor memory: T1 [0,128) T2 [128,256) P [256,320) dS [320,384)
// ACC1 [384,448) ACC2 [448,512). Every wait is bounded as in the forward.
//
// Head_dim 128: a 128-row tile is two 64-column swizzled boxes, and the
// score-shaped products take eight K-steps over both. dV and dK of 128
// columns would not fit beside S^T, dP^T, P and dS in the 512 columns of
// tensor memory, so a key-pass item also names a half of the head dimension:
// it computes S^T and dP^T over all 128 dimensions and accumulates only its
// 64 columns of dV and dK (the plan counts two items per key block and head).
// The query pass needs no P, so its dQ accumulator takes 128 columns
// [384,512). Two streaming stages of 64 KiB, and the epilogues store their
// rows directly (no staging), so shared memory stays within bounds. No
// two-head items.
// With local attention an item streams only the blocks inside the window band
// (key pass: the queries that can see its keys; query pass: the keys its rows
// can see) and the elementwise step zeroes P outside each row's window.
// Without a window, a sequence of at most 64 tokens runs two heads per item:
// every 128-row tile holds head h's rows in rows 0-63 and head h+1's in rows
// 64-127 (two 64-row TMA boxes), so each product's two diagonal 64x64 blocks
// are the two heads' and the elementwise step zeroes P and dS in the other two;
// the accumulations then need no change.
#pragma once

#include <cudaTypedefs.h>

#include "pe_kernels.cuh"
#include "pe_sm103.cuh"

namespace pe {

namespace {

using namespace sm103;

constexpr int kRows = 128;
constexpr int kThreads = 512;
// Registers per thread: 128 at launch (one CTA of 512 threads per SM); the
// producer/issuer warpgroups drop to kRegsLow and the two elementwise
// warpgroups rise to kRegsHigh, which holds a whole 64-column half-block of S
// and dP in registers.
constexpr uint32_t kRegsLaunch = 65536 / kThreads;
constexpr uint32_t kRegsLow = 56, kRegsHigh = 200;
static_assert(2 * 128 * (kRegsLow + kRegsHigh) <= kThreads * kRegsLaunch,
              "register split exceeds the launch allocation");
constexpr uint32_t kColT1 = 0, kColT2 = 128, kColP = 256, kColDS = 320, kColAcc1 = 384,
                   kColAcc2 = 448;
constexpr uint32_t kBoxBytes = kRows * 64 * 2;       // one 64-column swizzled box of a tile

// Shapes that depend on the head dimension D.
template <int D>
struct Cfg {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static constexpr int kStages = D == 64 ? 3 : 2;     // streaming tile pairs in flight
  static constexpr int kBoxes = D / 64;               // 64-column boxes per tile
  static constexpr int kHalves = D / 64;              // key-pass items per key block and head
  static constexpr uint32_t kTileBytes = kRows * D * 2;
  static constexpr bool kStagedStores = D == 64;      // TMA-store epilogue
};

struct Item {
  // head: in the key pass of head_dim 128, head * 2 + the half of the head
  // dimension (64 columns of dV and dK) that the item accumulates.
  int32_t seq, head, blk;
  int32_t dual;  // rows 0-63 of every tile are head `head`, rows 64-127 head + 1
};
constexpr uint32_t kHalfTileBytes = kRows * 64 * 2 / 2;  // 64 rows of a head_dim-64 tile

// Output staging: the 32 rows x 32 columns of each accumulator that an
// elementwise warp writes (2 KiB each, 64-byte swizzled), stored by TMA.
constexpr uint32_t kStageAccBytes = 32 * 32 * 2;

template <int D>
struct alignas(1024) Smem {
  static constexpr int kStages = Cfg<D>::kStages;
  __nv_bfloat16 st[2][kRows * D];              // stationary tiles
  __nv_bfloat16 u[kStages][2][kRows * D];      // streaming tile pairs
  float vec[kStages][2][kRows];                // key pass: -lse*log2e and -Delta per query column
  // Per elementwise warp: acc1, acc2 (head_dim 64; 128 stores directly).
  alignas(1024) uint8_t ostage[Cfg<D>::kStagedStores ? 8 : 1][2 * kStageAccBytes];
  uint64_t item_full[2], item_empty[2];
  uint64_t st_full, st_empty;
  uint64_t u_full[kStages], u_empty[kStages];
  uint64_t t_full[2], t_free;
  uint64_t p_full, acc_done[2];
  uint64_t o_full, o_free;
  uint64_t drain[4];
  Item items[2];
  uint32_t tmem_base;
  WaitGuard guard;
};

struct BwdParams {
  const int32_t* cu;
  int32_t B, H;
  int32_t pair_heads_rows;     // sequences up to this long run two heads per item (0: never)
  int64_t Nq;                  // lse / Delta row stride (= N)
  float scale, scale_log2;
  const float* lse;            // [H, N], natural log
  const float* delta;          // [H, N]
  __nv_bfloat16* out1;         // key pass: dK; query pass: dQ
  __nv_bfloat16* out2;         // key pass: dV
  TilePlan plan;
  Window win;
  DeviceStatus* status;
  uint64_t wait_limit_ns;   // bounded-wait limit of this launch
};

// The nblk streaming blocks of 128 rows of the item block `blk` of a sequence
// of len rows, the first one starting at row position org: in the key pass the
// query rows that see one of the item's keys, in the query pass the keys that
// one of the item's rows sees (the whole sequence without a window; with one
// the blocks start at the first row of the band, as TMA rows need no
// alignment). Never empty: a key is visible from its own position.
template <bool kKeyPass, bool kLocal>
__device__ __forceinline__ void stream_blocks(const BwdParams& p, int32_t len, int32_t blk,
                                              int32_t& org, int32_t& nblk) {
  if (!kLocal) {
    org = 0;
    nblk = (len + kRows - 1) / kRows;
    return;
  }
  const Window w = kKeyPass ? Window{p.win.right, p.win.left} : p.win;
  const int32_t first = blk * kRows, last = min(first + kRows, len) - 1;
  org = window_lo(w, first);
  nblk = (window_hi(w, last, len) - org) / kRows + 1;
}

enum WaitSite { kSiteProducer = 11, kSiteT = 12, kSiteAcc = 13, kSiteEw = 14 };

// kLocal selects the local-attention variant (block ranges and window masks);
// full attention compiles without them.
template <int D, bool kKeyPass, bool kLocal>
__global__ void __launch_bounds__(kThreads, 1)
bwd_sm103_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                 const __grid_constant__ CUtensorMap tm_q64,
                 const __grid_constant__ CUtensorMap tm_k64,
                 const __grid_constant__ CUtensorMap tm_v64,
                 const __grid_constant__ CUtensorMap tm_do64,
                 const __grid_constant__ CUtensorMap tm_o1,
                 const __grid_constant__ CUtensorMap tm_o2, const BwdParams p) {
  constexpr int kAccWarps = kKeyPass ? 2 : 1;
  constexpr int kUseWarps = 2 + kAccWarps;     // warps reading each streaming pair
  constexpr int kStages = Cfg<D>::kStages;
  constexpr int kBoxes = Cfg<D>::kBoxes;
  constexpr int kHalves = kKeyPass ? Cfg<D>::kHalves : 1;
  constexpr uint32_t kTileBytes = Cfg<D>::kTileBytes;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  Smem<D>& S =
      *reinterpret_cast<Smem<D>*>(smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile WaitGuard* abort_flag = &S.guard;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&S.item_full[i]), 1);
      mbar_init(smem_u32(&S.item_empty[i]), 1 + 2 + kAccWarps + 8);  // producer, issuers, elementwise
      mbar_init(smem_u32(&S.t_full[i]), 1);
      mbar_init(smem_u32(&S.acc_done[i]), 1);
    }
    mbar_init(smem_u32(&S.st_full), 1);
    mbar_init(smem_u32(&S.st_empty), 2);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&S.u_full[s]), kKeyPass ? 1 + 32 : 1);
      mbar_init(smem_u32(&S.u_empty[s]), kUseWarps);
    }
    mbar_init(smem_u32(&S.t_free), 8);
    mbar_init(smem_u32(&S.p_full), 8);
    mbar_init(smem_u32(&S.o_full), kAccWarps);
    mbar_init(smem_u32(&S.o_free), 8);
    for (int w = 0; w < 4; ++w) mbar_init(smem_u32(&S.drain[w]), 1);
    S.guard.abort = 0;
    S.guard.limit_ns = p.wait_limit_ns;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&S.tmem_base), 512);
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

  // Every role walks the same item sequence through the two-slot ring.
  auto read_item = [&](uint32_t item_no, Item& it, int site) -> bool {
    const int slot = item_no & 1;
    if (!warp_wait(smem_u32(&S.item_full[slot]), (item_no >> 1) & 1, abort_flag, p.status, site))
      return false;
    it = S.items[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&S.item_empty[slot]));
    return true;
  };

  // Warps 0-7 (producer, issuers, idle) hand registers to the elementwise
  // warpgroups; each warpgroup's setmaxnreg heads its own branch.
  if (warp < 8) {
    regs_release<kRegsLow>();
    if (warp == 0) {
      // ------------------------------------------------------------ producer (whole warp)
      const CUtensorMap* st_map0 = kKeyPass ? &tm_k : &tm_q;
      const CUtensorMap* st_map1 = kKeyPass ? &tm_v : &tm_do;
      const CUtensorMap* u_map0 = kKeyPass ? &tm_q : &tm_k;
      const CUtensorMap* u_map1 = kKeyPass ? &tm_do : &tm_v;
      // 64-row boxes for two-head items.
      const CUtensorMap* st_half0 = kKeyPass ? &tm_k64 : &tm_q64;
      const CUtensorMap* st_half1 = kKeyPass ? &tm_v64 : &tm_do64;
      const CUtensorMap* u_half0 = kKeyPass ? &tm_q64 : &tm_k64;
      const CUtensorMap* u_half1 = kKeyPass ? &tm_do64 : &tm_v64;
      if (lane == 0) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_do);
      }
      uint32_t u_no = 0;
      int pending_st = -1, pending_u[kStages];
      for (int s = 0; s < kStages; ++s) pending_u[s] = -1;
      bool ok = true;
      for (uint32_t item_no = 0; ok; ++item_no) {
        Item it;
        if (!read_item(item_no, it, kSiteProducer)) {
          ok = false;
          break;
        }
        if (it.seq < 0) break;
        const int32_t start = __ldg(p.cu + it.seq);
        const int32_t len = __ldg(p.cu + it.seq + 1) - start;
        int32_t org, nb;
        stream_blocks<kKeyPass, kLocal>(p, len, it.blk, org, nb);
        const int32_t x = (it.head / kHalves) * D;
        if (!warp_wait(smem_u32(&S.st_empty), (item_no & 1) ^ 1, abort_flag, p.status,
                       kSiteProducer)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(smem_u32(&S.st_full), 2 * kTileBytes);
          if (it.dual) {
            for (int hh = 0; hh < 2; ++hh) {
              tma_load_2d(smem_u32(S.st[0]) + hh * kHalfTileBytes, st_half0, smem_u32(&S.st_full),
                          x + hh * D, start);
              tma_load_2d(smem_u32(S.st[1]) + hh * kHalfTileBytes, st_half1, smem_u32(&S.st_full),
                          x + hh * D, start);
            }
          } else {
            for (int b = 0; b < kBoxes; ++b) {
              tma_load_2d(smem_u32(S.st[0]) + b * kBoxBytes, st_map0, smem_u32(&S.st_full),
                          x + 64 * b, start + it.blk * kRows);
              tma_load_2d(smem_u32(S.st[1]) + b * kBoxBytes, st_map1, smem_u32(&S.st_full),
                          x + 64 * b, start + it.blk * kRows);
            }
          }
        }
        pending_st = item_no & 1;
        for (int32_t i = 0; i < nb; ++i, ++u_no) {
          const int s = u_no % kStages;
          const uint32_t ph = (u_no / kStages) & 1;
          if (!warp_wait(smem_u32(&S.u_empty[s]), ph ^ 1, abort_flag, p.status, kSiteProducer)) {
            ok = false;
            break;
          }
          // The tiles first, then (key pass) the block's lse and Delta: the
          // global loads of those then overlap the copy instead of delaying it.
          // The stage completes on the copy's bytes and the 32 lanes' arrivals.
          if (lane == 0) {
            mbar_arrive_expect_tx(smem_u32(&S.u_full[s]), 2 * kTileBytes);
            if (it.dual) {
              for (int hh = 0; hh < 2; ++hh) {
                tma_load_2d(smem_u32(S.u[s][0]) + hh * kHalfTileBytes, u_half0,
                            smem_u32(&S.u_full[s]), x + hh * D, start);
                tma_load_2d(smem_u32(S.u[s][1]) + hh * kHalfTileBytes, u_half1,
                            smem_u32(&S.u_full[s]), x + hh * D, start);
              }
            } else {
              for (int b = 0; b < kBoxes; ++b) {
                tma_load_2d(smem_u32(S.u[s][0]) + b * kBoxBytes, u_map0, smem_u32(&S.u_full[s]),
                            x + 64 * b, start + org + i * kRows);
                tma_load_2d(smem_u32(S.u[s][1]) + b * kBoxBytes, u_map1, smem_u32(&S.u_full[s]),
                            x + 64 * b, start + org + i * kRows);
              }
            }
          }
          if (kKeyPass) {
            // -lse*log2e and -Delta of the block's 128 queries; -inf / 0 past
            // the sequence end, so those columns get P = 0.
            // A two-head item's columns 0-63 are head `head`'s queries at
            // positions 0-63, columns 64-127 head + 1's.
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int r = lane + 32 * u;
              const int32_t pos = it.dual ? (r & 63) : org + i * kRows + r;
              const int32_t hd = it.dual ? it.head + (r >> 6) : it.head / kHalves;
              const int64_t idx = static_cast<int64_t>(hd) * p.Nq + start + pos;
              const bool in = pos < len;
              S.vec[s][0][r] = in ? -__ldg(p.lse + idx) * kLog2e : -INFINITY;
              S.vec[s][1][r] = in ? -__ldg(p.delta + idx) : 0.f;
            }
          }
          if (kKeyPass) mbar_arrive(smem_u32(&S.u_full[s]));
          pending_u[s] = static_cast<int>(ph);
        }
      }
      if (!ok && lane == 0) {
        if (pending_st >= 0) mbar_drain_wait(smem_u32(&S.st_full), static_cast<uint32_t>(pending_st));
        for (int s = 0; s < kStages; ++s)
          if (pending_u[s] >= 0) mbar_drain_wait(smem_u32(&S.u_full[s]), static_cast<uint32_t>(pending_u[s]));
      }
    } else if (warp == 1 || warp == 2) {
      // ------------------------------------------------------------ score-shaped products
      // warp 1: T1 = A0 B0^T (S^T = K Q_i^T or S = Q K_j^T); warp 2: T2 = A1 B1^T (dP).
      const int w = warp - 1;
      constexpr uint32_t idesc = idesc_bf16(kRows, kRows, false, false);
      const uint32_t a_addr = smem_u32(S.st[w]);
      uint32_t u_no = 0, n_t = 0;
      bool ok = true;
      for (uint32_t item_no = 0; ok; ++item_no) {
        Item it;
        if (!read_item(item_no, it, kSiteT)) break;
        if (it.seq < 0) break;
        const int32_t len = __ldg(p.cu + it.seq + 1) - __ldg(p.cu + it.seq);
        int32_t org, nb;
        stream_blocks<kKeyPass, kLocal>(p, len, it.blk, org, nb);
        if (!warp_wait(smem_u32(&S.st_full), item_no & 1, abort_flag, p.status, kSiteT)) break;
        for (int32_t i = 0; i < nb; ++i, ++u_no, ++n_t) {
          const int s = u_no % kStages;
          if (!warp_wait(smem_u32(&S.u_full[s]), (u_no / kStages) & 1, abort_flag, p.status,
                         kSiteT) ||
              (n_t > 0 && !warp_wait(smem_u32(&S.t_free), (n_t - 1) & 1, abort_flag, p.status,
                                     kSiteT))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t b_addr = smem_u32(S.u[s][w]);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            // K-step kk: 16 columns of box kk / 4.
            const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
            mma_ss_warp(tmem + (w == 0 ? kColT1 : kColT2), smem_desc_sw128(a_addr + off, 16, 1024),
                        smem_desc_sw128(b_addr + off, 16, 1024), idesc, kk > 0 ? 1u : 0u);
          }
          tc_commit_warp(smem_u32(&S.t_full[w]));
          tc_commit_warp(smem_u32(&S.u_empty[s]));
        }
        if (ok) tc_commit_warp(smem_u32(&S.st_empty));
      }
      tc_commit_warp(smem_u32(&S.drain[w]));
      mbar_drain_wait(smem_u32(&S.drain[w]), 0);
    } else if (warp == 5) {
      // ------------------------------------------------------------ scheduler (whole warp)
      for (uint32_t item_no = 0;; ++item_no) {
        const int slot = item_no & 1;
        if (!warp_wait(smem_u32(&S.item_empty[slot]), ((item_no >> 1) & 1) ^ 1, abort_flag,
                       p.status, kSiteProducer))
          break;
        int32_t claimed = -1;
        if (lane == 0) {
          Item it;
          const int32_t t = atomicAdd(p.plan.counter, 1);
          if (t >= total) {
            it.seq = -1;
            it.head = it.blk = it.dual = 0;
          } else {
            int32_t seq, local;
            plan_decode(p.plan.order, p.plan.tile_end, p.B, t, seq, local);
            const int32_t len = __ldg(p.cu + seq + 1) - __ldg(p.cu + seq);
            it.seq = seq;
            if (len <= p.pair_heads_rows) {  // local indexes pairs of heads
              it.head = 2 * local;
              it.blk = 0;
              it.dual = it.head + 1 < p.H;
            } else {
              // With head_dim 128 the key pass's plan counts each head twice
              // (two halves of the head dimension): it.head is head * 2 + half.
              const int32_t nb = (len + kRows - 1) / kRows;
              it.head = local / nb;
              it.blk = local - it.head * nb;
              it.dual = 0;
            }
          }
          S.items[slot] = it;
          mbar_arrive(smem_u32(&S.item_full[slot]));
          claimed = it.seq;
        }
        if (__shfl_sync(0xffffffffu, claimed, 0) < 0) break;
      }
    } else if (warp == 3 || (kKeyPass && warp == 4)) {
      // ------------------------------------------------------------ accumulations
      // key pass: warp 3 dV += P^T dO_i, warp 4 dK += dS^T Q_i;
      // query pass: warp 3 dQ += dS K_j.
      const int w = warp - 3;
      constexpr uint32_t idesc = idesc_bf16(kRows, 64, false, true);  // N = 64 per MMA
      const uint32_t a_col = (kKeyPass && w == 0) ? kColP : kColDS;
      const uint32_t d_col = w == 0 ? kColAcc1 : kColAcc2;
      // The B operand: dO_i (dV), Q_i (dK) in the key pass; K_j in the query pass.
      const int b_idx = kKeyPass ? (w == 0 ? 1 : 0) : 0;
      uint32_t u_no = 0, n_p = 0;
      bool ok = true;
      for (uint32_t item_no = 0; ok; ++item_no) {
        Item it;
        if (!read_item(item_no, it, kSiteAcc)) break;
        if (it.seq < 0) break;
        const int32_t len = __ldg(p.cu + it.seq + 1) - __ldg(p.cu + it.seq);
        int32_t org, nb;
        stream_blocks<kKeyPass, kLocal>(p, len, it.blk, org, nb);
        // The previous item's accumulators must have been read by the epilogue.
        if (!warp_wait(smem_u32(&S.o_free), (item_no & 1) ^ 1, abort_flag, p.status, kSiteAcc))
          break;
        for (int32_t i = 0; i < nb; ++i, ++u_no, ++n_p) {
          const int s = u_no % kStages;
          if (!warp_wait(smem_u32(&S.u_full[s]), (u_no / kStages) & 1, abort_flag, p.status,
                         kSiteAcc) ||
              !warp_wait(smem_u32(&S.p_full), n_p & 1, abort_flag, p.status, kSiteAcc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // Key pass: the item's 64 columns (its half's box); query pass: all D
          // columns of dQ, one N = 64 MMA per box.
          const uint32_t b_addr =
              smem_u32(S.u[s][b_idx]) + (kHalves > 1 ? (it.head % kHalves) * kBoxBytes : 0u);
          constexpr int kN64 = kKeyPass ? 1 : kBoxes;
#pragma unroll
          for (int kk = 0; kk < kRows / 16; ++kk)
#pragma unroll
            for (int nh = 0; nh < kN64; ++nh)
              mma_ts_warp(tmem + d_col + 64 * nh, tmem + a_col + kk * 8,
                          smem_desc_sw128(b_addr + nh * kBoxBytes + kk * 16 * 128, 16, 1024),
                          idesc, (i > 0 || kk > 0) ? 1u : 0u);
          tc_commit_warp(smem_u32(&S.acc_done[w]));
          tc_commit_warp(smem_u32(&S.u_empty[s]));
        }
        if (ok) tc_commit_warp(smem_u32(&S.o_full));
      }
      tc_commit_warp(smem_u32(&S.drain[2 + w]));
      mbar_drain_wait(smem_u32(&S.drain[2 + w]), 0);
    }
  } else {
    regs_claim<kRegsHigh>();
    // ------------------------------------------------------------ elementwise + epilogue
    const int h = (warp - 8) >> 2;                // column half
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;          // tile row = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float scale_log2 = p.scale_log2;
    uint32_t u_no = 0, n_blk = 0, o_cnt = 0;
    bool ok = true;
    for (uint32_t item_no = 0; ok; ++item_no) {
      Item it;
      if (!read_item(item_no, it, kSiteEw)) break;
      if (it.seq < 0) break;
      const int32_t start = __ldg(p.cu + it.seq);
      const int32_t len = __ldg(p.cu + it.seq + 1) - start;
      int32_t org, nb;
      stream_blocks<kKeyPass, kLocal>(p, len, it.blk, org, nb);
      const int32_t r0 = it.blk * kRows;
      // This thread's row: in a two-head item rows 64-127 are head + 1's rows
      // at positions 0-63, and the column half that is the other head's is
      // off the diagonal (P = dS = 0 there).
      const bool off_diag = it.dual && (row >> 6) != h;  // warp-uniform
      // Streaming positions this row pairs with inside the window: the queries
      // that see this key (key pass) or the keys this query sees (query pass).
      constexpr bool windowed = kLocal;
      const Window wrow = kKeyPass ? Window{p.win.right, p.win.left} : p.win;
      const int32_t vis_lo = window_lo(wrow, r0 + row), vis_hi = window_hi(wrow, r0 + row, len);
      // Query pass: this thread's query row carries its own lse and Delta.
      // Off the diagonal of a two-head item an infinite lse makes P = 0.
      float row_lse2 = 0.f, row_delta = 0.f;
      if (!kKeyPass && (it.dual ? (row & 63) : r0 + row) < len) {
        const int64_t idx = static_cast<int64_t>(it.dual ? it.head + (row >> 6) : it.head) * p.Nq +
                            start + (it.dual ? (row & 63) : r0 + row);
        row_lse2 = off_diag ? INFINITY : __ldg(p.lse + idx) * kLog2e;
        row_delta = __ldg(p.delta + idx);
      }
      for (int32_t i = 0; i < nb; ++i, ++u_no, ++n_blk) {
        const int s = u_no % kStages;
        if (!warp_wait(smem_u32(&S.t_full[0]), n_blk & 1, abort_flag, p.status, kSiteEw) ||
            !warp_wait(smem_u32(&S.t_full[1]), n_blk & 1, abort_flag, p.status, kSiteEw) ||
            (kKeyPass && !warp_wait(smem_u32(&S.u_full[s]), (u_no / kStages) & 1, abort_flag,
                                    p.status, kSiteEw))) {
          ok = false;
          break;
        }
        tc_fence_after();
        // This half's 64 columns of both products into registers at once, so
        // that the next block's products can overwrite them while P and dS
        // are computed.
        uint32_t sv[2][32], dv[2][32];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          tmem_ld32(lane_base + kColT1 + 64 * h + 32 * c, sv[c]);
          tmem_ld32(lane_base + kColT2 + 64 * h + 32 * c, dv[c]);
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          tmem_wait_ld(sv[c]);
          tmem_wait_ld(dv[c]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&S.t_free));
        // Row position of this half's column 0.
        const int32_t col0_pos = it.dual ? 0 : org + i * kRows + 64 * h;
        const int32_t col_valid = len - col0_pos;           // query pass: valid keys in this half
        const int32_t clo = vis_lo - col0_pos, chi = vis_hi - col0_pos;  // window, same origin
        // Scores that must give P = 0 become -inf: keys past the sequence end
        // (query pass, the sequence's last block only; the key pass gets them
        // from the -inf lse of queries past the end) and pairs outside the window.
        if (kKeyPass && off_diag) {  // (the query pass gets P = 0 from its row's lse)
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int cc = 0; cc < 32; ++cc) sv[c][cc] = 0xff800000u;
        } else if (!kKeyPass && col_valid < 64) {
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int cc = 0; cc < 32; ++cc)
              if (32 * c + cc >= col_valid) sv[c][cc] = 0xff800000u;
        }
        if (windowed && __any_sync(0xffffffffu, clo > 0 || chi < 63)) {
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int cc = 0; cc < 32; ++cc)
              if (32 * c + cc < clo || 32 * c + cc > chi) sv[c][cc] = 0xff800000u;
        }
        uint32_t pk[2][16], dk[2][16];
        const uint64_t c2 = f2(scale_log2, scale_log2);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int col0 = 64 * h + 32 * c;
          // Key pass: -lse*log2e and -Delta per query column, four at a time;
          // query pass: this row's own.
          const float4* nl4 = reinterpret_cast<const float4*>(&S.vec[s][0][col0]);
          const float4* nd4 = reinterpret_cast<const float4*>(&S.vec[s][1][col0]);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            uint64_t nl2, nd2;
            if (kKeyPass) {
              const float4 l4 = nl4[e >> 1], d4 = nd4[e >> 1];
              nl2 = (e & 1) ? f2(l4.z, l4.w) : f2(l4.x, l4.y);
              nd2 = (e & 1) ? f2(d4.z, d4.w) : f2(d4.x, d4.y);
            } else {
              nl2 = f2(-row_lse2, -row_lse2);
              nd2 = f2(-row_delta, -row_delta);
            }
            float x0, x1;
            f2_split(ffma2(f2(__uint_as_float(sv[c][2 * e]), __uint_as_float(sv[c][2 * e + 1])),
                           c2, nl2),
                     x0, x1);
            const float pr[2] = {ex2(x0), ex2(x1)};
            const uint64_t g2 =
                fadd2(f2(__uint_as_float(dv[c][2 * e]), __uint_as_float(dv[c][2 * e + 1])), nd2);
            float ds0, ds1;
            f2_split(fmul2(f2(pr[0], pr[1]), g2), ds0, ds1);
            pk[c][e] = pack_bf16x2(pr[0], pr[1]);
            dk[c][e] = pack_bf16x2(ds0, ds1);
          }
        }
        // P and dS of the previous block must have been consumed before they are rewritten.
        if (n_blk > 0) {
          const uint32_t par = (n_blk - 1) & 1;
          if (!warp_wait(smem_u32(&S.acc_done[0]), par, abort_flag, p.status, kSiteEw) ||
              (kKeyPass && !warp_wait(smem_u32(&S.acc_done[1]), par, abort_flag, p.status,
                                      kSiteEw))) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          if (kKeyPass) tmem_st16(lane_base + kColP + 32 * h + 16 * c, pk[c]);
          tmem_st16(lane_base + kColDS + 32 * h + 16 * c, dk[c]);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&S.p_full));
      }
      if (!ok) break;
      // Epilogue: this half stores columns [32h, 32h+32) of dV and dK (the
      // item's 64), or columns [h*D/2, (h+1)*D/2) of dQ, in 32-column chunks.
      constexpr int kChunks = kKeyPass ? 1 : D / 64;
      if (!warp_wait(smem_u32(&S.o_full), o_cnt & 1, abort_flag, p.status, kSiteEw)) break;
      ++o_cnt;
      tc_fence_after();
      uint32_t a1[kChunks][32], a2[32];
#pragma unroll
      for (int c = 0; c < kChunks; ++c)
        tmem_ld32(lane_base + kColAcc1 + (kKeyPass ? 32 * h : (D / 2) * h + 32 * c), a1[c]);
#pragma unroll
      for (int c = 0; c < kChunks; ++c) tmem_wait_ld(a1[c]);
      if (kKeyPass) {
        tmem_ld32(lane_base + kColAcc2 + 32 * h, a2);
        tmem_wait_ld(a2);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&S.o_free));
      const int32_t pos_r = it.dual ? (row & 63) : r0 + row;
      const int32_t head_r = it.dual ? it.head + (row >> 6) : it.head / kHalves;
      // key pass: acc1 = dV (unscaled), acc2 = dK (times scale); query pass: acc1 = dQ * scale.
      const float s1 = kKeyPass ? 1.f : p.scale, s2 = p.scale;
      // A warp's 32 rows are 32 consecutive tokens of one head: when all are
      // real, its 32 columns of each accumulator go through a 64-byte-swizzled
      // stage to one TMA store; the partial warp at a sequence's end stores its
      // rows itself.
      const int32_t pos0 = pos_r - lane;               // warp-uniform
      // Global column of this thread's first chunk.
      const int32_t col0 =
          head_r * D + (kKeyPass ? (it.head % kHalves) * 64 + 32 * h : (D / 2) * h);
      if (Cfg<D>::kStagedStores && len - pos0 >= 32) {
        uint8_t* stage = S.ostage[warp - 8];
        if (lane == 0) bulk_wait_read();               // the previous stores have left the stage
        __syncwarp();
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const uint32_t off = lane * 64 + ((g ^ ((lane >> 1) & 3)) << 4);
          uint4 wv;
          wv.x = pack_bf16x2(__uint_as_float(a1[0][8 * g + 0]) * s1, __uint_as_float(a1[0][8 * g + 1]) * s1);
          wv.y = pack_bf16x2(__uint_as_float(a1[0][8 * g + 2]) * s1, __uint_as_float(a1[0][8 * g + 3]) * s1);
          wv.z = pack_bf16x2(__uint_as_float(a1[0][8 * g + 4]) * s1, __uint_as_float(a1[0][8 * g + 5]) * s1);
          wv.w = pack_bf16x2(__uint_as_float(a1[0][8 * g + 6]) * s1, __uint_as_float(a1[0][8 * g + 7]) * s1);
          *reinterpret_cast<uint4*>(stage + off) = wv;
          if (kKeyPass) {
            wv.x = pack_bf16x2(__uint_as_float(a2[8 * g + 0]) * s2, __uint_as_float(a2[8 * g + 1]) * s2);
            wv.y = pack_bf16x2(__uint_as_float(a2[8 * g + 2]) * s2, __uint_as_float(a2[8 * g + 3]) * s2);
            wv.z = pack_bf16x2(__uint_as_float(a2[8 * g + 4]) * s2, __uint_as_float(a2[8 * g + 5]) * s2);
            wv.w = pack_bf16x2(__uint_as_float(a2[8 * g + 6]) * s2, __uint_as_float(a2[8 * g + 7]) * s2);
            *reinterpret_cast<uint4*>(stage + kStageAccBytes + off) = wv;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int32_t x = col0, y = start + pos0;
          tma_store_2d(kKeyPass ? &tm_o2 : &tm_o1, smem_u32(stage), x, y);
          if (kKeyPass) tma_store_2d(&tm_o1, smem_u32(stage) + kStageAccBytes, x, y);
          bulk_commit();
        }
      } else if (pos_r < len) {
        const int64_t tok = static_cast<int64_t>(start) + pos_r;
        const int64_t off = tok * p.H * D + col0;
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
          uint4* d1 = reinterpret_cast<uint4*>((kKeyPass ? p.out2 : p.out1) + off + 32 * c);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint4 wv;
            wv.x = pack_bf16x2(__uint_as_float(a1[c][8 * g + 0]) * s1,
                               __uint_as_float(a1[c][8 * g + 1]) * s1);
            wv.y = pack_bf16x2(__uint_as_float(a1[c][8 * g + 2]) * s1,
                               __uint_as_float(a1[c][8 * g + 3]) * s1);
            wv.z = pack_bf16x2(__uint_as_float(a1[c][8 * g + 4]) * s1,
                               __uint_as_float(a1[c][8 * g + 5]) * s1);
            wv.w = pack_bf16x2(__uint_as_float(a1[c][8 * g + 6]) * s1,
                               __uint_as_float(a1[c][8 * g + 7]) * s1);
            d1[g] = wv;
          }
        }
        if (kKeyPass) {
          uint4* d2 = reinterpret_cast<uint4*>(p.out1 + off);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint4 wv;
            wv.x = pack_bf16x2(__uint_as_float(a2[8 * g + 0]) * s2, __uint_as_float(a2[8 * g + 1]) * s2);
            wv.y = pack_bf16x2(__uint_as_float(a2[8 * g + 2]) * s2, __uint_as_float(a2[8 * g + 3]) * s2);
            wv.z = pack_bf16x2(__uint_as_float(a2[8 * g + 4]) * s2, __uint_as_float(a2[8 * g + 5]) * s2);
            wv.w = pack_bf16x2(__uint_as_float(a2[8 * g + 6]) * s2, __uint_as_float(a2[8 * g + 7]) * s2);
            d2[g] = wv;
          }
        }
      }
    }
    bulk_wait_all();                                   // every row is written before the CTA retires
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode_bwd = nullptr;

pe_status get_encoder_bwd() {
  if (g_encode_bwd) return PE_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult qres;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &qres) != cudaSuccess ||
      qres != cudaDriverEntryPointSuccess || !fn)
    return PE_ERR_CUDA;
  g_encode_bwd = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return PE_OK;
}

// [N, H*D] bf16 rows, loaded as boxes of 64 columns (128 bytes, the swizzle
// span) and box_rows rows.
template <int D>
pe_status make_map_bwd(CUtensorMap* map, const void* base, int64_t N, int32_t H,
                       uint32_t box_rows = kRows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(H) * D, static_cast<cuuint64_t>(N)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * D * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t elem_strides[2] = {1, 1};
  CUresult r = g_encode_bwd(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
                            dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PE_OK : PE_ERR_CUDA;
}

// [N, H*D] bf16 gradient rows; stores of 32 rows x 32 columns, 64-byte swizzle
// (used by the head_dim-64 epilogue).
template <int D>
pe_status make_map_out(CUtensorMap* map, void* base, int64_t N, int32_t H) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(H) * D, static_cast<cuuint64_t>(N)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * D * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t elem_strides[2] = {1, 1};
  CUresult r = g_encode_bwd(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box,
                            elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PE_OK : PE_ERR_CUDA;
}

template <int D, bool kKeyPass>
pe_status launch_pass(const CUtensorMap (&m)[8], const BwdParams& prm, LayoutCheck check,
                      cudaStream_t stream) {
  // Output maps: key pass dK (out1) and dV (out2), query pass dQ (out1).
  CUtensorMap mo1, mo2;
  PE_TRY(make_map_out<D>(&mo1, prm.out1, prm.Nq, prm.H));
  PE_TRY(make_map_out<D>(&mo2, kKeyPass ? prm.out2 : prm.out1, prm.Nq, prm.H));
  auto kernel = prm.win.active() ? bwd_sm103_kernel<D, kKeyPass, true>
                                 : bwd_sm103_kernel<D, kKeyPass, false>;
  const size_t smem = sizeof(Smem<D>) + 1024;
  PE_CUDA_TRY(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(smem)));
  // The elementwise warpgroups' register claim is served from what the CTA
  // was launched with; never launch a build whose count cannot serve it.
  cudaFuncAttributes attr;
  PE_CUDA_TRY(cudaFuncGetAttributes(&attr, kernel));
  if (static_cast<uint32_t>(attr.numRegs) * kThreads < 2u * 128u * (kRegsLow + kRegsHigh))
    return PE_ERR_UNSUPPORTED;
  // The key pass counts each head once per half of the head dimension.
  PE_TRY(launch_tile_plan(prm.cu, prm.B, kKeyPass ? prm.H * Cfg<D>::kHalves : prm.H, kRows,
                          prm.pair_heads_rows, 0, prm.plan, check, stream));
  PE_TRY(launch_after_previous(kernel, dim3(device_sm_count()), dim3(kThreads), smem, stream,
                               m[0], m[1], m[2], m[3], m[4], m[5], m[6], m[7], mo1, mo2, prm));
  PE_CUDA_TRY(cudaGetLastError());
  return PE_OK;
}

// Both passes; Delta = rowsum(dO o O) is already in `delta`.
template <int D>
pe_status bwd_sm103_impl(const void* q, const void* k, const void* v, const int32_t* cu,
                         int32_t B, int32_t H, int64_t N, float scale, Window win,
                         const float* lse, const void* dout, const float* delta, void* dq,
                         void* dk, void* dv, TilePlan plan, LayoutCheck check,
                         cudaStream_t stream) {
  PE_TRY(get_encoder_bwd());
  // q, k, v, dO with 128-row boxes, then with 64-row boxes (two-head items).
  CUtensorMap maps[8];
  const void* bases[4] = {q, k, v, dout};
  for (int m = 0; m < 8; ++m)
    PE_TRY(make_map_bwd<D>(&maps[m], bases[m % 4], N, H, m < 4 ? kRows : 64));
  BwdParams prm;
  prm.cu = cu;
  prm.B = B;
  prm.H = H;
  prm.pair_heads_rows = (win.active() || D != 64) ? 0 : 64;
  prm.Nq = N;
  prm.scale = scale;
  prm.scale_log2 = scale * kLog2e;
  prm.win = win;
  prm.lse = lse;
  prm.delta = delta;
  prm.plan = plan;
  prm.status = check.status;
  prm.wait_limit_ns = wait_limit_ns();
  prm.out1 = static_cast<__nv_bfloat16*>(dk);
  prm.out2 = static_cast<__nv_bfloat16*>(dv);
  PE_TRY((launch_pass<D, true>(maps, prm, check, stream)));
  prm.out1 = static_cast<__nv_bfloat16*>(dq);
  prm.out2 = nullptr;
  return launch_pass<D, false>(maps, prm, check, stream);
}

}  // namespace
}  // namespace pe
