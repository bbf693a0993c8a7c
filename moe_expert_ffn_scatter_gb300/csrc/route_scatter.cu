// route_scatter.cu -- top-k routing, aligned prefix-sum endpoints and the
// token scatter with fused group-128 e4m3 / UE8M0 input quantisation.
//
// [LR] §2: the scatter writes the int32 endpoint of each expert inside the
// existing step, with no count read back to the host; start[e] =
// align_up(end[e-1], A), end[e] = start[e] + count[e].
// [DG] §2.2.4 (compact layout: per-token-group quantisation, ep_scatter into
// expert-contiguous segments) and 附录 C (src2dst).
//
// Three launches, all with grids fixed by (T, E, k, H) so a CUDA graph can
// replay them while routing changes:
//   1. route_count_kernel   one block per chunk of 64 tokens: routing (16
//      warps, one token per warp at a time), then one warp ranks the chunk's
//      routes per expert in row-major (token, slot) order with match_any and
//      writes the rank inside the chunk to src2dst and the chunk histogram to
//      the workspace.
//   2. endpoints_kernel     one block: per expert, exclusive prefix of the
//      chunk histograms (workspace becomes per-chunk row bases), block scan of
//      the A-aligned counts -> start/end, expert_ends written.
//   3. scatter_quant_kernel one warp per token: final src2dst, then the token
//      row is quantised once (16 lanes per 128-column group, uint4 loads) and
//      its codes and packed scale words are stored to each destination row.
#include <climits>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

// Routing of one token by one warp. Lane i holds logits e = i + 32 m.
template <int EPL, int MODE>
__device__ __forceinline__ void route_token(const float* __restrict__ l, const float* __restrict__ bias,
                                            int E, int k, int lane, int32_t* __restrict__ ids_out,
                                            float* __restrict__ w_out, int32_t* ids_smem) {
  float v[EPL];
  uint32_t removed = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    float s = 0.0f;
    if (e < E) {
      const float x = l[e];
      s = (MODE == MOE_ROUTE_SIGMOID_BIAS_TOPK) ? __fadd_rn(spec_sigmoid(x), bias[e]) : x;
    } else {
      removed |= 1u << i;
    }
    v[i] = s;
  }
  int my_idx = 0;
  for (int j = 0; j < k; ++j) {
    float bv = 0.0f;
    int bi = INT_MAX;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      if (!((removed >> i) & 1u) && (bi == INT_MAX || v[i] > bv)) {
        bv = v[i];
        bi = lane + 32 * i;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(kFull, bv, o);
      const int oi = __shfl_xor_sync(kFull, bi, o);
      if (oi != INT_MAX && (bi == INT_MAX || ov > bv || (ov == bv && oi < bi))) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) removed |= 1u << (bi >> 5);
    if (lane == j) my_idx = bi;
  }
  // Weights, slot j on lane j; sums run in slot order like the definition.
  const float lj = (lane < k) ? l[my_idx] : 0.0f;
  float num;
  if (MODE == MOE_ROUTE_SIGMOID_BIAS_TOPK) {
    num = (lane < k) ? spec_sigmoid(lj) : 0.0f;
  } else {
    const float m = __shfl_sync(kFull, lj, 0);
    num = (lane < k) ? spec_exp(__fsub_rn(lj, m)) : 0.0f;
  }
  float s = 0.0f;
  for (int j = 0; j < k; ++j) s = __fadd_rn(s, __shfl_sync(kFull, num, j));
  if (lane < k) {
    ids_out[lane] = my_idx;
    ids_smem[lane] = my_idx;
    w_out[lane] = __fdiv_rn(num, s);
  }
}

template <int EPL, int MODE>
__global__ void __launch_bounds__(512) route_count_kernel(const float* __restrict__ logits,
                                                          const float* __restrict__ bias,
                                                          int32_t* __restrict__ ids,
                                                          float* __restrict__ topw,
                                                          int32_t* __restrict__ s2d,
                                                          int32_t* __restrict__ ws, int T, int E,
                                                          int k) {
  extern __shared__ int32_t smem_i32[];
  int32_t* cnt = smem_i32;                 // [E] running count per expert
  int32_t* ids_s = smem_i32 + E;           // [kScatterChunk * k] the chunk's expert ids
  const int c = blockIdx.x;
  const int t0 = c * kScatterChunk;
  const int t1 = min(T, t0 + kScatterChunk);
  const int nr = (t1 - t0) * k;
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  if (MODE != MOE_ROUTE_PRECOMPUTED) {
    for (int t = t0 + warp; t < t1; t += nwarps)
      route_token<EPL, MODE>(logits + (size_t)t * E, bias, E, k, lane, ids + (size_t)t * k,
                             topw + (size_t)t * k, ids_s + (t - t0) * k);
  } else {
    for (int r = threadIdx.x; r < nr; r += blockDim.x) ids_s[r] = ids[(size_t)t0 * k + r];
  }
  __syncthreads();
  if (warp == 0) {
    // Stable rank of every route inside the chunk: routes in row-major
    // (token, slot) order, 32 at a time; peers with the same expert are ranked
    // by lane, then the group's count is added to the expert's running count.
    for (int base = 0; base < nr; base += 32) {
      const int r = base + lane;
      const int e = (r < nr) ? ids_s[r] : -1;
      const bool valid = (e >= 0 && e < E);
      const unsigned peers = __match_any_sync(kFull, valid ? e : -1);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int leader = __ffs(peers) - 1;
      const int before = valid ? cnt[e] : 0;
      __syncwarp();
      if (valid && lane == leader) cnt[e] = before + __popc(peers);
      __syncwarp();
      if (r < nr) s2d[(size_t)t0 * k + r] = valid ? before + rank : -1;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) ws[(size_t)c * E + e] = cnt[e];
}

// Endpoints. With `counts` given, count[e] = counts[e]; otherwise count[e] is
// the sum of the chunk histograms, which are replaced by per-chunk row bases
// (start[e] + routes of e in earlier chunks). One warp per expert scans the
// chunk histograms (lanes over chunks); the block then scans the A-aligned
// counts over experts.
__global__ void __launch_bounds__(1024) endpoints_kernel(const int32_t* __restrict__ counts,
                                                         int32_t* __restrict__ ws, int nchunks, int E,
                                                         int A, int32_t* __restrict__ ends, long cap,
                                                         uint32_t* err) {
  extern __shared__ int32_t cnt_s[];       // [E]
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t carry;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  if (threadIdx.x == 0) carry = 0;
  if (counts) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt_s[e] = counts[e];
  } else {
    for (int e = warp; e < E; e += nwarps) {
      int run = 0;
      for (int c0 = 0; c0 < nchunks; c0 += 32) {
        const int c = c0 + lane;
        const int v = (c < nchunks) ? ws[(size_t)c * E + e] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int n = __shfl_up_sync(kFull, incl, o);
          if (lane >= o) incl += n;
        }
        if (c < nchunks) ws[(size_t)c * E + e] = run + incl - v;
        run += __shfl_sync(kFull, incl, 31);
      }
      if (lane == 0) cnt_s[e] = run;
    }
  }
  __syncthreads();
  for (int base = 0; base < E; base += 1024) {
    const int e = base + threadIdx.x;
    const int total = (e < E) ? cnt_s[e] : 0;
    const int aligned = (e < E) ? (int)align_up64(total, A) : 0;
    int v = aligned;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(kFull, v, o);
      if (lane >= o) v += n;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int s = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, s, o);
        if (lane >= o) s += n;
      }
      warp_sums[lane] = s;
    }
    __syncthreads();
    const int start = carry + (v - aligned) + (warp > 0 ? warp_sums[warp - 1] : 0);
    if (e < E) {
      ends[e] = start + total;
      cnt_s[e] = start;  // reused below as the expert's start row
    }
    __syncthreads();
    if (threadIdx.x == 0) carry += warp_sums[31];
    __syncthreads();
  }
  if (!counts) {
    for (int e = warp; e < E; e += nwarps) {
      const int start = cnt_s[e];
      for (int c = lane; c < nchunks; c += 32) ws[(size_t)c * E + e] += start;
    }
  }
  if (threadIdx.x == 0 && E > 0 && cap >= 0 && (long)ends[E - 1] > cap) raise_error(err, MOE_DEVERR_CAPACITY);
}

__device__ __forceinline__ uint32_t e4m3x4(const float* f, float sc) {
  return e4m3x2_satfinite(__fmul_rn(f[0], sc), __fmul_rn(f[1], sc)) |
         (e4m3x2_satfinite(__fmul_rn(f[2], sc), __fmul_rn(f[3], sc)) << 16);
}

__global__ void __launch_bounds__(256) scatter_quant_kernel(const uint16_t* __restrict__ x,
                                                            const int32_t* __restrict__ ids,
                                                            int32_t* __restrict__ s2d,
                                                            const int32_t* __restrict__ ws,
                                                            uint8_t* __restrict__ a_fp8,
                                                            int32_t* __restrict__ a_sf, int T, int E,
                                                            int k, int H, int ld_sf, long cap,
                                                            uint32_t* err) {
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int G = H / 128;
  const int npass = (H + 255) / 256;
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += gridDim.x * wpb) {
    int dst = -1;
    if (lane < k) {
      const int e = ids[(size_t)t * k + lane];
      const int lr = s2d[(size_t)t * k + lane];
      if (e >= 0 && e < E && lr >= 0) {
        dst = ws[(size_t)(t / kScatterChunk) * E + e] + lr;
        if ((long)dst >= cap) {
          raise_error(err, MOE_DEVERR_CAPACITY);
          dst = -1;
        }
      }
      s2d[(size_t)t * k + lane] = dst;
    }
    const uint16_t* xr = x + (size_t)t * H;
    uint32_t word = 0;
    for (int it0 = 0; it0 < npass; it0 += 4) {
      uint4 v[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int col = (it0 + p) * 256 + lane * 8;
        v[p] = (col < H) ? __ldg(reinterpret_cast<const uint4*>(xr + col)) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int it = it0 + p;
        if (it >= npass) break;
        const int col = it * 256 + lane * 8;
        const bool active = col < H;
        float f[8];
        f[0] = bf16_lo(v[p].x); f[1] = bf16_hi(v[p].x);
        f[2] = bf16_lo(v[p].y); f[3] = bf16_hi(v[p].y);
        f[4] = bf16_lo(v[p].z); f[5] = bf16_hi(v[p].z);
        f[6] = bf16_lo(v[p].w); f[7] = bf16_hi(v[p].w);
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
        const uint32_t b = active ? group_scale_byte(amax) : 0u;
        const float sc = pow2_f32(127 - (int)b);
        uint2 codes;
        codes.x = e4m3x4(f, sc);
        codes.y = e4m3x4(f + 4, sc);
        for (int j = 0; j < k; ++j) {
          const int d = __shfl_sync(kFull, dst, j);
          if (d >= 0 && active) *reinterpret_cast<uint2*>(a_fp8 + (size_t)d * H + col) = codes;
        }
        const uint32_t b_lo = __shfl_sync(kFull, b, 0);
        const uint32_t b_hi = __shfl_sync(kFull, b, 16);
        const int g0 = 2 * it;
        word |= b_lo << (8 * (g0 & 3));
        if (g0 + 1 < G) word |= b_hi << (8 * ((g0 + 1) & 3));
        if (((g0 + 1) & 3) == 3 || g0 + 2 >= G) {
          if (dst >= 0) a_sf[(size_t)(g0 >> 2) * ld_sf + dst] = (int32_t)word;
          word = 0;
        }
      }
    }
  }
}

template <int EPL, int MODE>
cudaError_t launch_route_count(const moe_route_args& a, int nchunks, cudaStream_t st) {
  const size_t smem = (size_t)(a.E + kScatterChunk * a.k) * sizeof(int32_t);
  route_count_kernel<EPL, MODE><<<nchunks, 512, smem, st>>>(
      a.logits, a.corr_bias, a.topk_ids, a.topk_w, a.src2dst, (int32_t*)a.workspace, a.T, a.E, a.k);
  return cudaGetLastError();
}

template <int MODE>
cudaError_t dispatch_epl(const moe_route_args& a, int nchunks, cudaStream_t st) {
  const int epl = (a.E + 31) / 32;
  if (epl <= 1) return launch_route_count<1, MODE>(a, nchunks, st);
  if (epl <= 2) return launch_route_count<2, MODE>(a, nchunks, st);
  if (epl <= 4) return launch_route_count<4, MODE>(a, nchunks, st);
  if (epl <= 8) return launch_route_count<8, MODE>(a, nchunks, st);
  if (epl <= 16) return launch_route_count<16, MODE>(a, nchunks, st);
  return launch_route_count<32, MODE>(a, nchunks, st);
}

}  // namespace

size_t route_scatter_ws_bytes(int T, int E, int k) {
  (void)k;
  const size_t nchunks = (size_t)(T + kScatterChunk - 1) / kScatterChunk;
  const size_t b = nchunks * (size_t)E * sizeof(int32_t);
  return b < 16 ? 16 : (b + 15) / 16 * 16;
}

cudaError_t launch_expert_ends(const int32_t* counts, int E, int A, int32_t* ends, uint32_t* err,
                               cudaStream_t st) {
  endpoints_kernel<<<1, 1024, (size_t)E * sizeof(int32_t), st>>>(counts, nullptr, 0, E, A, ends, -1, err);
  return cudaGetLastError();
}

cudaError_t launch_route_scatter(const moe_route_args& a, int num_sms, uint32_t* err, cudaStream_t st) {
  const int nchunks = (a.T + kScatterChunk - 1) / kScatterChunk;
  cudaError_t ce = cudaSuccess;
  if (nchunks > 0) {
    if (a.routing_mode == MOE_ROUTE_SOFTMAX_TOPK)
      ce = dispatch_epl<MOE_ROUTE_SOFTMAX_TOPK>(a, nchunks, st);
    else if (a.routing_mode == MOE_ROUTE_SIGMOID_BIAS_TOPK)
      ce = dispatch_epl<MOE_ROUTE_SIGMOID_BIAS_TOPK>(a, nchunks, st);
    else
      ce = launch_route_count<1, MOE_ROUTE_PRECOMPUTED>(a, nchunks, st);
    if (ce != cudaSuccess) return ce;
  }
  endpoints_kernel<<<1, 1024, (size_t)a.E * sizeof(int32_t), st>>>(nullptr, (int32_t*)a.workspace, nchunks,
                                                                   a.E, a.A, a.expert_ends, a.cap, err);
  if ((ce = cudaGetLastError()) != cudaSuccess) return ce;
  if (a.T > 0) {
    const int blocks = (int)lmin((a.T + 7) / 8, (long)num_sms * 16);
    scatter_quant_kernel<<<blocks, 256, 0, st>>>(a.x, a.topk_ids, a.src2dst, (const int32_t*)a.workspace,
                                                 a.a_fp8, a.a_sf, a.T, a.E, a.k, a.H,
                                                 (int)align_up64(a.cap, 4), a.cap, err);
    ce = cudaGetLastError();
  }
  return ce;
}

// ---------------------------------------------------- no-allocation variant
// Scratch of moe_route_scatter_noalloc: the per-chunk expert histograms live
// in this file-scope device array instead of a caller-provided workspace.
// Every GPU that loads the library holds these 1 MiB until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
static __device__ __align__(256) int32_t g_route_scratch[kNoAllocScratchBytes / sizeof(int32_t)];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};
}  // namespace

size_t route_scatter_noalloc_max_bytes() { return kNoAllocScratchBytes; }

// `device` must be the current device. Its first call on a device looks the
// array's device address up once (the host-side symbol is only a stand-in,
// never a device address) and caches it.
cudaError_t launch_route_scatter_noalloc(const moe_route_args& a, int device, int num_sms, uint32_t* err,
                                         cudaStream_t st) {
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[device]) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
      if (e != cudaSuccess) return e;
      g_scratch_addr[device] = p;
    }
    scratch = g_scratch_addr[device];
  }
  moe_route_args b = a;
  b.workspace = scratch;
  b.workspace_bytes = kNoAllocScratchBytes;
  return launch_route_scatter(b, num_sms, err, st);
}

}  // namespace moe
