// First-token query, streaming backward.
//
// With one query row per sequence (its first token; page "Source code for
// gigl.nn.packed_attention", function `packed_attention`,
// `query_is_first_token`, and the custom op gigl::varlen_attention_backward
// that takes the saved output and log-sum-exp) the gradients of sequence i
// and head h of softmax attention follow row by row over its visible keys j:
//
//   P_j  = exp(scale q.k_j - lse)        dP_j = dO.v_j        Delta = dO.O
//   dS_j = P_j (dP_j - Delta)
//   dv_j = P_j dO      dk_j = scale dS_j q      dq = scale sum_j dS_j k_j
//
// Each key row is used by exactly one query, so dk and dv are written once per
// row, as soon as the row is read, and the cost is moving k and v in and dk
// and dv out (four token rows per key). The kernel streams whole rows through
// the ring of pe_token_stream.cuh (equal token chunks, one CTA each): the four
// consumer warps take the rows of each stage in turn; for every 16-byte vector
// of a row a lane forms its share of q.k and dO.v, the lanes of one head add
// their shares with xor shuffles (so they all hold the same sums), and the
// lane then writes its vectors of dv and dk and updates its dq sums. Rows of
// the chunk that the query does not see (beyond a window) get zero dk and dv.
//
// Delta is formed from the saved output that the op receives (in bf16 the
// exact output rounded), for dq and dk alike, so the result is the gradient
// formula evaluated with that saved output.
//
// dq: at a sequence's end in the chunk the warps' sums are added in shared
// memory (fixed warp order). A sequence inside one chunk is finished there; a
// sequence whose visible keys cross chunk edges leaves its chunk sum in one
// slot per chunk (slot 1 in its first chunk, slot 0 in the others) that
// first_token_bwd_merge_kernel adds in chunk order. No atomics: the results
// are bitwise reproducible.
//
// Supported when a token row is a whole number of 512-byte warp loads (bf16
// rows up to 3072 bytes, fp32 rows up to 4096: at most 48 and 32 elements per
// lane, which the one-CTA-per-SM register budget holds without spilling) and
// D is 32, 64 or 128; other shapes run the CUDA-core backward.
#include "pe_kernels.cuh"
#include "pe_token_stream.cuh"

namespace pe {
namespace {

using namespace stream;

enum BwdWaitSite { kSiteBwdProducer = 23, kSiteBwdConsumer = 24 };

template <typename T, int D, int VPL>
struct BwdShape : Shape<T, D, VPL> {
  using Base = Shape<T, D, VPL>;
  // Two CTAs per SM (at most 168 registers a thread: ten warps over four
  // schedulers) up to 24 elements of a row per lane; one (255) beyond, where
  // 168 would spill.
  static constexpr int kMinBlocks = VPL * Base::kEPV <= 24 ? 2 : 1;
  static constexpr size_t kSmem = Base::kRingBytes + (size_t)kWarps * Base::kRow * sizeof(float);
  static_assert(VPL * Base::kEPV <= 48, "at most 48 elements of a row per lane");
};

template <typename T, int D, int VPL>
__global__ void __launch_bounds__(kBlock, BwdShape<T, D, VPL>::kMinBlocks)
first_token_bwd_stream_kernel(const T* __restrict__ q, const T* __restrict__ k,
                              const T* __restrict__ v, const T* __restrict__ out,
                              const T* __restrict__ dout, const float* __restrict__ lse,
                              const int32_t* __restrict__ cu, int32_t B, int64_t N,
                              int32_t chunk, float scale, int32_t key_limit,
                              T* __restrict__ dq, T* __restrict__ dk, T* __restrict__ dv,
                              float* __restrict__ part, DeviceStatus* status,
                              uint64_t wait_limit_ns) {
  using Sh = BwdShape<T, D, VPL>;
  constexpr int EPV = Sh::kEPV, LPH = Sh::kLPH, ROW = Sh::kRow, R = Sh::kRows;
  constexpr int kUGroup = VPL < 4 ? VPL : 4;
  extern __shared__ __align__(128) unsigned char bw_smem[];
  T* ks = reinterpret_cast<T*>(bw_smem);                     // [stages][R][ROW]
  T* vs = ks + kStages * Sh::kStageElems;                    // [stages][R][ROW]
  float* s_dq = reinterpret_cast<float*>(vs + kStages * Sh::kStageElems);  // [warps][ROW]
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
  __shared__ WaitGuard guard;
  __shared__ int32_t entry_code;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t c0 = (int64_t)blockIdx.x * chunk;
  const int64_t c1 = min(N, c0 + chunk);
  // Launched behind the layout check: nothing it wrote (the status word) is
  // read before it has finished. The merge kernel may be scheduled meanwhile.
  griddep_wait();
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), kWarps);
    }
    guard.abort = 0;
    guard.limit_ns = wait_limit_ns;
    // Read once for the whole CTA: other CTAs may record a timeout meanwhile.
    entry_code = *reinterpret_cast<volatile int32_t*>(&status->code);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (entry_code != PE_OK) return;  // the layout failed its check: read nothing
  volatile WaitGuard* abort_flag = &guard;
  const int32_t first = find_sequence(cu, B, (int32_t)c0, lane);

  if (warp == kWarps) {
    if (lane == 0)
      produce_rows<Sh>(k, v, cu, first, c0, c1, key_limit, ks, vs, full, empty, abort_flag,
                       status, kSiteBwdProducer);
    return;
  }

  // A wait that gives up ends this warp's stage loop; the consumers then meet
  // at the dq barrier, which tells all of them whether any gave up, and leave
  // together without writing dq.
  const float scale_log2 = scale * kLog2e;
  uint32_t g = 0;  // stages consumed
  int32_t i = first;
  for (int64_t a = c0; a < c1; ++i) {
    const Segment sg = segment_of(cu, i, a, c1, key_limit);
    a = sg.next;
    // Rows of the chunk outside the query's window: zero gradients.
    for (int64_t row = max(sg.a, sg.vis_end) + warp; row < sg.next; row += kWarps) {
#pragma unroll
      for (int u = 0; u < VPL; ++u) {
        const int64_t off = row * ROW + (u * 32 + lane) * EPV;
        store16(dk + off, make_uint4(0u, 0u, 0u, 0u));
        store16(dv + off, make_uint4(0u, 0u, 0u, 0u));
      }
    }
    if (sg.a >= sg.vis_end) continue;  // CTA-uniform
    // The sequence's query row and output gradient (kept packed, widened on
    // use), Delta and lse (base 2) of this lane's heads.
    uint4 qp[VPL], dop[VPL];
    float delta[VPL], lse2[VPL];
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
      const int64_t off = (int64_t)i * ROW + (u * 32 + lane) * EPV;
      qp[u] = load16(q + off);
      dop[u] = load16(dout + off);
      float ov[EPV], dov[EPV];
      unpack16<T>(load16(out + off), ov);
      unpack16<T>(dop[u], dov);
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < EPV; ++e) d = fmaf(dov[e], ov[e], d);
#pragma unroll
      for (int x = 1; x < LPH; x <<= 1) d += __shfl_xor_sync(0xffffffffu, d, x);
      delta[u] = d;
      const int h = (u * 32 + lane) / LPH;
      lse2[u] = __ldg(lse + (int64_t)h * B + i) * kLog2e;
    }
    float acc[VPL][EPV];  // dq / scale
#pragma unroll
    for (int u = 0; u < VPL; ++u)
#pragma unroll
      for (int e = 0; e < EPV; ++e) acc[u][e] = 0.f;
    bool failed = false;
    for (int64_t r0 = sg.a; r0 < sg.vis_end; r0 += R, ++g) {
      const int s = g % kStages;
      // Every consumer warp waits for and releases every stage.
      if (!warp_wait(smem_u32(&full[s]), (g / kStages) & 1, abort_flag, status,
                     kSiteBwdConsumer)) {
        failed = true;
        break;
      }
      const int nr = (int)min((int64_t)R, sg.vis_end - r0);
      const T* kst = ks + s * Sh::kStageElems;
      const T* vst = vs + s * Sh::kStageElems;
      for (int r = warp; r < nr; r += kWarps) {
        T* dkr = dk + (r0 + r) * ROW;
        T* dvr = dv + (r0 + r) * ROW;
        // The row's vectors in groups of at most four (each vector's heads
        // reduce on their own), so that wide rows keep few values live
        // across the reductions.
#pragma unroll
        for (int ub = 0; ub < VPL; ub += kUGroup) {
          float sc[kUGroup], dp[kUGroup];
#pragma unroll
          for (int uu = 0; uu < kUGroup; ++uu) {
            const int u = ub + uu;
            if (u >= VPL) break;
            const int col = (u * 32 + lane) * EPV;
            float kx[EPV], vx[EPV], qx[EPV], dx[EPV];
            unpack16<T>(*reinterpret_cast<const uint4*>(kst + r * ROW + col), kx);
            unpack16<T>(*reinterpret_cast<const uint4*>(vst + r * ROW + col), vx);
            unpack16<T>(qp[u], qx);
            unpack16<T>(dop[u], dx);
            float s1 = 0.f, s2 = 0.f;
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
              s1 = fmaf(qx[e], kx[e], s1);
              s2 = fmaf(dx[e], vx[e], s2);
            }
            sc[uu] = s1;
            dp[uu] = s2;
          }
#pragma unroll
          for (int x = 1; x < LPH; x <<= 1) {
#pragma unroll
            for (int uu = 0; uu < kUGroup; ++uu) {
              if (ub + uu >= VPL) break;
              sc[uu] += __shfl_xor_sync(0xffffffffu, sc[uu], x);
              dp[uu] += __shfl_xor_sync(0xffffffffu, dp[uu], x);
            }
          }
#pragma unroll
          for (int uu = 0; uu < kUGroup; ++uu) {
            const int u = ub + uu;
            if (u >= VPL) break;
            const int col = (u * 32 + lane) * EPV;
            const float p = ex2(fmaf(sc[uu], scale_log2, -lse2[u]));
            const float ds = p * (dp[uu] - delta[u]);
            const float dss = ds * scale;
            float kx[EPV], qx[EPV], dx[EPV], gv[EPV], gk[EPV];
            unpack16<T>(*reinterpret_cast<const uint4*>(kst + r * ROW + col), kx);
            unpack16<T>(qp[u], qx);
            unpack16<T>(dop[u], dx);
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
              gv[e] = p * dx[e];
              gk[e] = dss * qx[e];
              acc[u][e] = fmaf(ds, kx[e], acc[u][e]);
            }
            store16(dvr + col, pack16<T>(gv));
            store16(dkr + col, pack16<T>(gk));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    }
    // Add the warps' sums: each thread takes ROW / threads elements.
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
      const int col = (u * 32 + lane) * EPV;
#pragma unroll
      for (int e = 0; e < EPV; ++e) s_dq[warp * ROW + col + e] = acc[u][e];
    }
    if (consumers_sync_or(failed)) return;
    const bool whole = sg.s0 >= c0 && sg.e1 <= c1;
    float* slot = part + ((int64_t)blockIdx.x * 2 + (sg.s0 < c0 ? 0 : 1)) * ROW;
    for (int idx = threadIdx.x; idx < ROW; idx += kThreads) {
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) sum += s_dq[w * ROW + idx];
      if (whole)
        dq[(int64_t)i * ROW + idx] = from_f32<T>(sum * scale);
      else
        slot[idx] = sum;
    }
    consumers_sync();  // s_dq free for the next sequence
  }
}

// One warp per (sequence, head) whose visible keys cross a chunk edge: adds
// its chunk sums in chunk order, four chunks' loads in flight at a time.
template <typename T, int D>
__global__ void first_token_bwd_merge_kernel(const float* __restrict__ part,
                                             const int32_t* __restrict__ cu, int32_t B,
                                             int32_t H, int32_t chunk, int32_t key_limit,
                                             float scale, T* __restrict__ dq,
                                             const DeviceStatus* __restrict__ status) {
  griddep_wait();  // launched behind the streaming kernel: its chunk sums are complete
  // An invalid layout or a streaming kernel that gave up: nothing to add.
  if (status->code != PE_OK) return;
  constexpr int kU = 4;
  constexpr int kC = D / 32;  // columns per lane: lane, lane + 32, ...
  static_assert(D % 32 == 0, "whole columns per lane");
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)H * D;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t ih = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
       ih < (int64_t)B * H; ih += warps) {
    const int32_t i = (int32_t)(ih / H), h = (int32_t)(ih - (int64_t)i * H);
    const int64_t s0 = __ldg(cu + i), s1 = __ldg(cu + i + 1);
    const int64_t e1 = min(s1, s0 + key_limit);
    const int64_t cb = s0 / chunk, ce = (e1 - 1) / chunk;
    if (cb == ce) continue;  // finished by the streaming kernel
    float sum[kC];
#pragma unroll
    for (int j = 0; j < kC; ++j) sum[j] = 0.f;
    for (int64_t c = cb; c <= ce; c += kU) {
      float x[kU][kC];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int64_t cc = c + u;
        const float* p = part + (cc * 2 + (cc == cb ? 1 : 0)) * row + (int64_t)h * D;
#pragma unroll
        for (int j = 0; j < kC; ++j) x[u][j] = cc <= ce ? __ldg(p + lane + 32 * j) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kU; ++u)
#pragma unroll
        for (int j = 0; j < kC; ++j) sum[j] += x[u][j];
    }
#pragma unroll
    for (int j = 0; j < kC; ++j)
      dq[ih * D + lane + 32 * j] = from_f32<T>(sum[j] * scale);
  }
}

template <typename T, int D, int VPL>
pe_status launch_bwd(const void* q, const void* k, const void* v, const void* out,
                     const void* dout, const float* lse, const int32_t* cu, int32_t B, int32_t H,
                     int64_t N, int32_t chunk, float scale, int32_t key_limit, void* dq, void* dk,
                     void* dv, float* part, DeviceStatus* status, cudaStream_t stream) {
  using Sh = BwdShape<T, D, VPL>;
  const auto kernel = first_token_bwd_stream_kernel<T, D, VPL>;
  PE_CUDA_TRY(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)Sh::kSmem));
  // One wave of equal token ranges, never shorter than the workspace's chunk
  // (so the chunk sums always fit).
  chunk = (int32_t)max((int64_t)chunk, ceil_div(N, (int64_t)device_sm_count() * Sh::kMinBlocks));
  const int64_t blocks = ceil_div(N, chunk);
  PE_TRY(launch_after_previous(kernel, dim3((unsigned)blocks), dim3(kBlock), Sh::kSmem, stream,
                               static_cast<const T*>(q), static_cast<const T*>(k),
                               static_cast<const T*>(v), static_cast<const T*>(out),
                               static_cast<const T*>(dout), lse, cu, B, N, chunk, scale,
                               key_limit, static_cast<T*>(dq), static_cast<T*>(dk),
                               static_cast<T*>(dv), part, status, wait_limit_ns()));
  int64_t mblocks = ceil_div((int64_t)B * H, 8);
  const int64_t cap = (int64_t)device_sm_count() * 16;
  if (mblocks > cap) mblocks = cap;
  PE_TRY(launch_after_previous(first_token_bwd_merge_kernel<T, D>, dim3((unsigned)mblocks),
                               dim3(256), 0, stream, static_cast<const float*>(part), cu, B, H,
                               chunk, key_limit, scale, static_cast<T*>(dq),
                               static_cast<const DeviceStatus*>(status)));
  return PE_OK;
}

template <typename T, int D>
pe_status dispatch_vpl(int vpl, const void* q, const void* k, const void* v, const void* out,
                       const void* dout, const float* lse, const int32_t* cu, int32_t B,
                       int32_t H, int64_t N, int32_t chunk, float scale, int32_t key_limit,
                       void* dq, void* dk, void* dv, float* part, DeviceStatus* status,
                       cudaStream_t stream) {
  constexpr int kMaxVpl = sizeof(T) == 4 ? 8 : 6;
  switch (vpl) {
#define PE_CASE(n)                                                                          \
  case n:                                                                                   \
    if constexpr (n <= kMaxVpl)                                                             \
      return launch_bwd<T, D, n>(q, k, v, out, dout, lse, cu, B, H, N, chunk, scale,         \
                                 key_limit, dq, dk, dv, part, status, stream);               \
    return PE_ERR_UNSUPPORTED;
    PE_CASE(1) PE_CASE(2) PE_CASE(3) PE_CASE(4) PE_CASE(5) PE_CASE(6) PE_CASE(7) PE_CASE(8)
#undef PE_CASE
    default: return PE_ERR_UNSUPPORTED;
  }
}

template <typename T>
pe_status dispatch_d(int D, int vpl, const void* q, const void* k, const void* v,
                     const void* out, const void* dout, const float* lse, const int32_t* cu,
                     int32_t B, int32_t H, int64_t N, int32_t chunk, float scale,
                     int32_t key_limit, void* dq, void* dk, void* dv, float* part,
                     DeviceStatus* status, cudaStream_t stream) {
  switch (D) {
#define PE_D(d)                                                                           \
  case d:                                                                                 \
    return dispatch_vpl<T, d>(vpl, q, k, v, out, dout, lse, cu, B, H, N, chunk, scale,    \
                              key_limit, dq, dk, dv, part, status, stream);
    PE_D(32) PE_D(64) PE_D(128)
#undef PE_D
    default: return PE_ERR_UNSUPPORTED;
  }
}

int bwd_vectors_per_lane(pe_dtype dtype, int32_t H, int32_t D) {
  const int vpl = vectors_per_lane(dtype, H, D);
  return vpl >= 1 && vpl <= (dtype == PE_FP32 ? 8 : 6) ? vpl : 0;
}

}  // namespace

bool first_token_bwd_stream_supported(pe_dtype dtype, int32_t H, int32_t D) {
  return (D == 32 || D == 64 || D == 128) && bwd_vectors_per_lane(dtype, H, D) > 0;
}

size_t first_token_bwd_stream_partial_bytes(int64_t N, int32_t H, int32_t D) {
  const int64_t chunks = ceil_div(N, first_token_stream_chunk(N));
  return ((size_t)chunks * 2 * H * D * sizeof(float) + 15) / 16 * 16;
}

pe_status bwd_first_token_stream(pe_dtype dtype, int32_t D, const void* q, const void* k,
                                 const void* v, const void* out, const void* dout,
                                 const float* lse, const int32_t* cu, int32_t B, int32_t H,
                                 int64_t N, int32_t S, float scale, Window win, void* dq,
                                 void* dk, void* dv, float* part, DeviceStatus* status,
                                 cudaStream_t stream) {
  const int vpl = bwd_vectors_per_lane(dtype, H, D);
  if (!vpl || !part) return PE_ERR_UNSUPPORTED;
  // With a window the query at position 0 sees keys 0 .. right.
  const int32_t key_limit = win.right == kUnbounded ? S : min(S, win.right + 1);
  const int32_t chunk = first_token_stream_chunk(N);
  if (dtype == PE_FP32)
    return dispatch_d<float>(D, vpl, q, k, v, out, dout, lse, cu, B, H, N, chunk, scale,
                             key_limit, dq, dk, dv, part, status, stream);
  return dispatch_d<__nv_bfloat16>(D, vpl, q, k, v, out, dout, lse, cu, B, H, N, chunk, scale,
                                   key_limit, dq, dk, dv, part, status, stream);
}

}  // namespace pe
