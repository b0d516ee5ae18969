// First-token query, streaming forward.
//
// In first-token mode every sequence has one query row (its first token), so
// the forward is a matrix-vector product per (sequence, head) whose cost is
// reading k and v once (page "Source code for gigl.nn.packed_attention",
// function `packed_attention`, `query_is_first_token`). The kernel streams
// whole token rows through the ring of pe_token_stream.cuh (equal token
// chunks, one CTA each, a producer thread and four consumer warps):
//
//  * the consumers keep one online-softmax state per (lane, vector), release
//    each stage, and at each sequence's end merge their states in shared
//    memory;
//  * a sequence that lies inside one chunk is finished there (output, lse); a
//    sequence that crosses chunk edges leaves one partial state (m, l, o[D]
//    per head) in every chunk it touches (slot 1 in its first chunk, slot 0
//    in the others), which first_token_stream_merge_kernel combines in chunk
//    order. Nothing is accumulated with atomics, so results are bitwise
//    reproducible.
//
// Supported when a token row is a whole number (1..8) of 512-byte warp loads
// and a head's row slice spans a power of two of lanes (D in {32, 64, 128});
// other shapes run the per-(sequence, head) kernel in pe_fwd_simt.cu.
#include "pe_kernels.cuh"
#include "pe_token_stream.cuh"

namespace pe {
namespace {

using namespace stream;

constexpr int kStWarps = stream::kWarps;
constexpr int kStThreads = stream::kThreads;
constexpr int kStBlock = stream::kBlock;
constexpr int kStStages = stream::kStages;
constexpr int32_t kStMaxChunks = 16384;
enum StWaitSite { kSiteStProducer = 21, kSiteStConsumer = 22 };

template <typename T, int D, int VPL>
struct StShape : Shape<T, D, VPL> {
  static constexpr int kMinBlocks = VPL <= 6 ? 2 : 1;
  static constexpr size_t kSmem =
      Shape<T, D, VPL>::kRingBytes +
      (size_t)kStWarps * (Shape<T, D, VPL>::kRow + 2 * Shape<T, D, VPL>::kH) * sizeof(float);
};

// Partial state of (chunk c, slot, head h): m, l, o[D].
template <int D>
__device__ __forceinline__ float* partial_state(float* part, int64_t c, int slot, int H, int h) {
  return part + ((c * 2 + slot) * H + h) * (D + 2);
}

template <typename T, int D, int VPL>
__global__ void __launch_bounds__(kStBlock, StShape<T, D, VPL>::kMinBlocks)
first_token_stream_kernel(const T* __restrict__ q, const T* __restrict__ k,
                          const T* __restrict__ v, const int32_t* __restrict__ cu, int32_t B,
                          int64_t N, int32_t chunk, float scale_log2, int32_t key_limit,
                          T* __restrict__ out, float* __restrict__ lse, float* __restrict__ part,
                          DeviceStatus* status, uint64_t wait_limit_ns) {
  using Sh = StShape<T, D, VPL>;
  constexpr int EPV = Sh::kEPV, LPH = Sh::kLPH, ROW = Sh::kRow, H = Sh::kH, R = Sh::kRows;
  extern __shared__ __align__(128) unsigned char st_smem[];
  T* ks = reinterpret_cast<T*>(st_smem);                       // [stages][R][ROW]
  T* vs = ks + kStStages * Sh::kStageElems;                    // [stages][R][ROW]
  float* s_o = reinterpret_cast<float*>(vs + kStStages * Sh::kStageElems);  // [warps][ROW]
  float* s_m = s_o + kStWarps * ROW;                           // [warps][H]
  float* s_l = s_m + kStWarps * H;                             // [warps][H]
  __shared__ __align__(8) uint64_t full[kStStages], empty[kStStages];
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
    for (int s = 0; s < kStStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), kStWarps);
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

  if (warp == kStWarps) {
    if (lane == 0)
      produce_rows<Sh>(k, v, cu, first, c0, c1, key_limit, ks, vs, full, empty, abort_flag,
                       status, kSiteStProducer);
    return;
  }

  // -------------------------------------------------------------- consumers
  // A wait that gives up ends this warp's stage loop; the consumers then meet
  // at the merge barrier, which tells all of them whether any gave up, and
  // leave together without writing anything (so no warp is left waiting at a
  // barrier that a departed warp would never reach).
  uint32_t g = 0;  // stages consumed
  int32_t i = first;
  for (int64_t a = c0; a < c1; ++i) {
    const Segment sg = segment_of(cu, i, a, c1, key_limit);
    a = sg.next;
    if (sg.a >= sg.vis_end) continue;  // CTA-uniform
    float qv[VPL][EPV];
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
      unpack16<T>(load16(q + (int64_t)i * ROW + (u * 32 + lane) * EPV), qv[u]);
#pragma unroll
      for (int e = 0; e < EPV; ++e) qv[u][e] *= scale_log2;
    }
    bool failed = false;
    float m[VPL], l[VPL], o[VPL][EPV];
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
      m[u] = -INFINITY;
      l[u] = 0.f;
#pragma unroll
      for (int e = 0; e < EPV; ++e) o[u][e] = 0.f;
    }
    for (int64_t r0 = sg.a; r0 < sg.vis_end; r0 += R, ++g) {
      const int s = g % kStStages;
      // Every consumer warp waits for and releases every stage.
      if (!warp_wait(smem_u32(&full[s]), (g / kStStages) & 1, abort_flag, status,
                     kSiteStConsumer)) {
        failed = true;
        break;
      }
      const int nr = (int)min((int64_t)R, sg.vis_end - r0);
      const T* kst = ks + s * Sh::kStageElems;
      const T* vst = vs + s * Sh::kStageElems;
      for (int r = warp; r < nr; r += kStWarps) {
        float sc[VPL];
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
          float kx[EPV];
          unpack16<T>(*reinterpret_cast<const uint4*>(kst + r * ROW + (u * 32 + lane) * EPV),
                      kx);
          float d = 0.f;
#pragma unroll
          for (int e = 0; e < EPV; ++e) d = fmaf(qv[u][e], kx[e], d);
#pragma unroll
          for (int off = 1; off < LPH; off <<= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
          sc[u] = d;
        }
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
          const float mx = fmaxf(m[u], sc[u]);
          const float corr = ex2(m[u] - mx);  // 0 on the first row
          const float p = ex2(sc[u] - mx);
          float vx[EPV];
          unpack16<T>(*reinterpret_cast<const uint4*>(vst + r * ROW + (u * 32 + lane) * EPV),
                      vx);
          l[u] = fmaf(l[u], corr, p);
#pragma unroll
          for (int e = 0; e < EPV; ++e) o[u][e] = fmaf(p, vx[e], o[u][e] * corr);
          m[u] = mx;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    }
    // Merge the warps' states: each thread combines ROW / threads elements.
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
      const int col = (u * 32 + lane) * EPV;
#pragma unroll
      for (int e = 0; e < EPV; ++e) s_o[warp * ROW + col + e] = o[u][e];
      if (lane % LPH == 0) {
        const int h = (u * 32 + lane) / LPH;
        s_m[warp * H + h] = m[u];
        s_l[warp * H + h] = l[u];
      }
    }
    if (consumers_sync_or(failed)) return;
    const int64_t s0 = sg.s0, e1 = sg.e1;
    const bool whole = s0 >= c0 && e1 <= c1;
    const int slot = s0 < c0 ? 0 : 1;
    for (int idx = threadIdx.x; idx < ROW; idx += kStThreads) {
      const int h = idx / D, col = idx - h * D;
      float gm = -INFINITY;
#pragma unroll
      for (int w = 0; w < kStWarps; ++w) gm = fmaxf(gm, s_m[w * H + h]);
      float gl = 0.f, go = 0.f;
#pragma unroll
      for (int w = 0; w < kStWarps; ++w) {
        const float lw = s_l[w * H + h];
        const float wt = lw > 0.f ? ex2(s_m[w * H + h] - gm) : 0.f;
        gl = fmaf(lw, wt, gl);
        go = fmaf(s_o[w * ROW + idx], wt, go);
      }
      if (whole) {
        out[(int64_t)i * ROW + idx] = from_f32<T>(go / gl);
        if (lse && col == 0) lse[(int64_t)h * B + i] = (gm + __log2f(gl)) * kLn2;
      } else {
        float* p = partial_state<D>(part, blockIdx.x, slot, H, h);
        p[2 + col] = go;
        if (col == 0) {
          p[0] = gm;
          p[1] = gl;
        }
      }
    }
    consumers_sync();  // s_o, s_m, s_l free for the next sequence
  }
}


// One warp per (sequence, head) whose visible keys cross a chunk edge:
// combines its partials in chunk order, m = max m_c, l = sum l_c 2^(m_c - m),
// o = sum o_c 2^(m_c - m) / l. Lanes take partials (for m and l) or columns
// (for o); loads are issued sixteen partials at a time.
template <typename T, int D>
__global__ void first_token_stream_merge_kernel(const float* __restrict__ part,
                                                const int32_t* __restrict__ cu, int32_t B,
                                                int32_t H, int32_t chunk, int32_t key_limit,
                                                T* __restrict__ out, float* __restrict__ lse,
                                                const DeviceStatus* __restrict__ status) {
  griddep_wait();  // launched behind the streaming kernel: its partials are complete
  // An invalid layout or a streaming kernel that gave up: nothing to combine.
  if (status->code != PE_OK) return;
  constexpr int kU = 16;
  static_assert(D % 32 == 0, "whole columns per lane");
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t ih = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
       ih < (int64_t)B * H; ih += warps) {
    const int32_t i = (int32_t)(ih / H), h = (int32_t)(ih - (int64_t)i * H);
    const int64_t s0 = __ldg(cu + i), s1 = __ldg(cu + i + 1);
    const int64_t e1 = min(s1, s0 + key_limit);
    const int64_t cb = s0 / chunk, ce = (e1 - 1) / chunk;
    if (cb == ce) continue;  // finished by the streaming kernel
    auto state = [&](int64_t c) {
      return part + ((c * 2 + (c == cb ? 1 : 0)) * H + h) * (D + 2);
    };
    float gm = -INFINITY;
    for (int64_t c = cb + lane; c <= ce; c += 32) gm = fmaxf(gm, state(c)[0]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, off));
    float gl = 0.f;
    for (int64_t c = cb + lane; c <= ce; c += 32) {
      const float* p = state(c);
      if (p[1] > 0.f) gl = fmaf(p[1], ex2(p[0] - gm), gl);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) gl += __shfl_xor_sync(0xffffffffu, gl, off);
    constexpr int kC = D / 32;  // columns per lane: lane, lane + 32, ...
    float go[kC];
#pragma unroll
    for (int j = 0; j < kC; ++j) go[j] = 0.f;
    for (int64_t c = cb; c <= ce; c += kU) {
      float mc[kU], lc[kU], oc[kU][kC];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        lc[u] = 0.f;
        mc[u] = 0.f;
#pragma unroll
        for (int j = 0; j < kC; ++j) oc[u][j] = 0.f;
        if (c + u <= ce) {
          const float* p = state(c + u);
          mc[u] = p[0];
          lc[u] = p[1];
#pragma unroll
          for (int j = 0; j < kC; ++j) oc[u][j] = p[2 + lane + 32 * j];
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const float w = lc[u] > 0.f ? ex2(mc[u] - gm) : 0.f;
#pragma unroll
        for (int j = 0; j < kC; ++j) go[j] = fmaf(oc[u][j], w, go[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < kC; ++j)
      out[((int64_t)i * H + h) * D + lane + 32 * j] = from_f32<T>(go[j] / gl);
    if (lse && lane == 0) lse[(int64_t)h * B + i] = (gm + __log2f(gl)) * kLn2;
  }
}

template <typename T, int D, int VPL>
pe_status launch_stream(const void* q, const void* k, const void* v, const int32_t* cu,
                        int32_t B, int32_t H, int64_t N, int32_t chunk, float scale,
                        int32_t key_limit, void* out, float* lse, float* part,
                        DeviceStatus* status, cudaStream_t stream) {
  using Sh = StShape<T, D, VPL>;
  const auto kernel = first_token_stream_kernel<T, D, VPL>;
  PE_CUDA_TRY(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)Sh::kSmem));
  // One wave of equal token ranges: every CTA resident at once moves the same
  // bytes, and long sequences leave few partials. The range never falls below
  // the workspace's chunk, so the partials always fit.
  chunk = (int32_t)max((int64_t)chunk,
                       ceil_div(N, (int64_t)device_sm_count() * Sh::kMinBlocks));
  const int64_t blocks = ceil_div(N, chunk);
  PE_TRY(launch_after_previous(kernel, dim3((unsigned)blocks), dim3(kStBlock), Sh::kSmem, stream,
                               static_cast<const T*>(q), static_cast<const T*>(k),
                               static_cast<const T*>(v), cu, B, N, chunk, scale * kLog2e,
                               key_limit, static_cast<T*>(out), lse, part, status,
                               wait_limit_ns()));
  int64_t mblocks = ceil_div((int64_t)B * H, 8);
  const int64_t cap = (int64_t)device_sm_count() * 16;
  if (mblocks > cap) mblocks = cap;
  PE_TRY(launch_after_previous(first_token_stream_merge_kernel<T, D>, dim3((unsigned)mblocks),
                               dim3(256), 0, stream, static_cast<const float*>(part), cu, B, H,
                               chunk, key_limit, static_cast<T*>(out), lse,
                               static_cast<const DeviceStatus*>(status)));
  return PE_OK;
}

template <typename T, int D>
pe_status dispatch_vpl(int vpl, const void* q, const void* k, const void* v, const int32_t* cu,
                       int32_t B, int32_t H, int64_t N, int32_t chunk, float scale,
                       int32_t key_limit, void* out, float* lse, float* part,
                       DeviceStatus* status, cudaStream_t stream) {
  switch (vpl) {
#define PE_CASE(n)                                                                        \
  case n:                                                                                 \
    return launch_stream<T, D, n>(q, k, v, cu, B, H, N, chunk, scale, key_limit, out, lse, \
                                  part, status, stream);
    PE_CASE(1) PE_CASE(2) PE_CASE(3) PE_CASE(4) PE_CASE(5) PE_CASE(6) PE_CASE(7) PE_CASE(8)
#undef PE_CASE
    default: return PE_ERR_UNSUPPORTED;
  }
}

template <typename T>
pe_status dispatch_d(int D, int vpl, const void* q, const void* k, const void* v,
                     const int32_t* cu, int32_t B, int32_t H, int64_t N, int32_t chunk,
                     float scale, int32_t key_limit, void* out, float* lse, float* part,
                     DeviceStatus* status, cudaStream_t stream) {
  switch (D) {
    case 32:
      return dispatch_vpl<T, 32>(vpl, q, k, v, cu, B, H, N, chunk, scale, key_limit, out, lse,
                                 part, status, stream);
    case 64:
      return dispatch_vpl<T, 64>(vpl, q, k, v, cu, B, H, N, chunk, scale, key_limit, out, lse,
                                 part, status, stream);
    case 128:
      return dispatch_vpl<T, 128>(vpl, q, k, v, cu, B, H, N, chunk, scale, key_limit, out, lse,
                                  part, status, stream);
    default: return PE_ERR_UNSUPPORTED;
  }
}

int stream_vectors_per_lane(pe_dtype dtype, int32_t H, int32_t D) {
  const int vpl = vectors_per_lane(dtype, H, D);
  return vpl >= 1 && vpl <= 8 ? vpl : 0;
}

}  // namespace

bool first_token_stream_supported(pe_dtype dtype, int32_t H, int32_t D) {
  return (D == 32 || D == 64 || D == 128) && stream_vectors_per_lane(dtype, H, D) > 0;
}

int32_t first_token_stream_chunk(int64_t N) {
  int32_t chunk = 64;
  while (ceil_div(N, chunk) > kStMaxChunks) chunk *= 2;
  return chunk;
}

size_t first_token_stream_partial_bytes(int64_t N, int32_t H, int32_t D) {
  const int64_t chunks = ceil_div(N, first_token_stream_chunk(N));
  return ((size_t)chunks * 2 * H * (D + 2) * sizeof(float) + 15) / 16 * 16;
}

pe_status fwd_first_token_stream(pe_dtype dtype, int32_t D, const void* q, const void* k,
                                 const void* v, const int32_t* cu, int32_t B, int32_t H,
                                 int64_t N, int32_t S, float scale, Window win, void* out,
                                 float* lse, float* part, DeviceStatus* status,
                                 cudaStream_t stream) {
  const int vpl = stream_vectors_per_lane(dtype, H, D);
  if (!vpl || !part) return PE_ERR_UNSUPPORTED;
  // With a window the query at position 0 sees keys 0 .. right.
  const int32_t key_limit = win.right == kUnbounded ? S : min(S, win.right + 1);
  const int32_t chunk = first_token_stream_chunk(N);
  if (dtype == PE_FP32)
    return dispatch_d<float>(D, vpl, q, k, v, cu, B, H, N, chunk, scale, key_limit, out, lse,
                             part, status, stream);
  return dispatch_d<__nv_bfloat16>(D, vpl, q, k, v, cu, B, H, N, chunk, scale, key_limit, out,
                                   lse, part, status, stream);
}

}  // namespace pe
