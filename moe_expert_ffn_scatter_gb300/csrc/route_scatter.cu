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
//   1. route_kernel         one warp per token: scores -> selection keys, top-k
//      from per-lane sorted lists with warp max/min reductions, weights
//      (replaced by a 4-byte memset when the caller supplies the routing).
//   2. rank_count_kernel    one block per chunk of 64 tokens: one warp ranks
//      the chunk's routes per expert in row-major (token, slot) order with
//      match_any; rank inside the chunk -> src2dst, chunk histogram ->
//      workspace. The last block to finish then computes the endpoints: per
//      expert, exclusive prefix of the chunk histograms over chunks
//      (coalesced, independent loads), then a block scan of the A-aligned
//      counts -> expert_ends (endpoints_block; endpoints_kernel runs the same
//      code alone for counts given by the caller, or T = 0).
//   3. scatter_quant_kernel one warp per token: final src2dst = start[e] +
//      chunk prefix + rank, then the token row is quantised once (16 lanes per
//      128-column group, or 4 per 32-column group in the MXFP8 recipe; uint4
//      loads) and its codes and packed scale words are stored to each
//      destination row.
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "pipeline.cuh"

namespace moe {

namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

// Selection key of a routing score: a larger score has a larger key, +0 and
// -0 share one key (they compare equal), NaN ranks below every number. Key 0
// marks an entry that cannot be selected (already chosen, or e >= E).
__device__ __forceinline__ uint32_t score_key(float s) {
  if (s != s) return 1u;
  uint32_t b = __float_as_uint(s);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The lane's LN best selectable entries, best first. Slots are visited in
// increasing order; a new entry goes in front of the first strictly smaller
// key and the entries behind it move down one, so equal keys stay in slot
// (= expert index) order.
template <int EPL, int LN>
__device__ __forceinline__ void build_list(const uint32_t (&key)[EPL], uint32_t removed, uint32_t (&lk)[LN],
                                           int (&li)[LN]) {
#pragma unroll
  for (int p = 0; p < LN; ++p) {
    lk[p] = 0u;
    li[p] = 0;
  }
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    uint32_t kk = ((removed >> i) & 1u) ? 0u : key[i];
    int ii = i;
    bool shifting = false;  // once the entry is placed, the rest move down one
#pragma unroll
    for (int p = 0; p < LN; ++p) {
      const bool take = shifting || kk > lk[p];
      shifting = take;
      const uint32_t tk = lk[p];
      const int ti = li[p];
      lk[p] = take ? kk : tk;
      li[p] = take ? ii : ti;
      kk = take ? tk : kk;
      ii = take ? ti : ii;
    }
  }
}

// Routing of one token by one warp. Lane i holds the scores of experts
// e = i + 32 m as selection keys and keeps its best LN of them in a short
// sorted list. Each of the k rounds takes the warp maximum of the list heads
// (redux), the lowest expert index among the lanes holding it, and advances
// the winner's list; a lane whose list runs dry rebuilds it from the entries
// not yet chosen. The result is the top-k in descending score, ties to the
// lower expert index.
template <int EPL, int MODE>
__device__ __forceinline__ void route_token(const float* __restrict__ l, const float* __restrict__ bias,
                                            int E, int k, int lane, int32_t* __restrict__ ids_out,
                                            float* __restrict__ w_out) {
  constexpr int LN = EPL < 4 ? EPL : 4;
  uint32_t key[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    uint32_t kk = 0u;
    if (e < E) {
      const float x = __ldg(l + e);
      kk = score_key((MODE == MOE_ROUTE_SIGMOID_BIAS_TOPK) ? __fadd_rn(spec_sigmoid(x), __ldg(bias + e)) : x);
    }
    key[i] = kk;
  }
  uint32_t removed = 0u;
  uint32_t lk[LN];
  int li[LN];
  build_list<EPL, LN>(key, removed, lk, li);
  int my_idx = 0;
  for (int j = 0; j < k; ++j) {
    const uint32_t gmax = __reduce_max_sync(kFull, lk[0]);
    const int cand = (lk[0] == gmax && gmax != 0u) ? lane + 32 * li[0] : INT_MAX;
    const int gidx = __reduce_min_sync(kFull, cand);
    if (lane == j) my_idx = gidx;
    if (cand == gidx) {
      removed |= 1u << li[0];
#pragma unroll
      for (int p = 0; p + 1 < LN; ++p) {
        lk[p] = lk[p + 1];
        li[p] = li[p + 1];
      }
      lk[LN - 1] = 0u;
      if (LN < EPL && lk[0] == 0u) build_list<EPL, LN>(key, removed, lk, li);
    }
  }
  // Weights, slot j on lane j; sums run in slot order like the definition.
  // (k <= E keeps a selectable entry in some list every round, so my_idx < E.)
  const float lj = (lane < k && my_idx < E) ? l[my_idx] : 0.0f;
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
    w_out[lane] = __fdiv_rn(num, s);
  }
}

// One warp per token over the whole grid.
// Block 0 also zeroes the completion count of the rank/count launch that
// follows (`done`, in the workspace).
template <int EPL, int MODE>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits,
                                                    const float* __restrict__ bias, int32_t* __restrict__ ids,
                                                    float* __restrict__ topw, int T, int E, int k,
                                                    unsigned int* __restrict__ done) {
  const int lane = threadIdx.x & 31;
  if (blockIdx.x == 0 && threadIdx.x == 0 && done) *done = 0u;
  const int wpb = blockDim.x >> 5;
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += gridDim.x * wpb)
    route_token<EPL, MODE>(logits + (size_t)t * E, bias, E, k, lane, ids + (size_t)t * k, topw + (size_t)t * k);
}

// One block per chunk of kScatterChunk tokens: the chunk's routes are ranked
// per expert in row-major (token, slot) order -- 32 at a time by one warp,
// peers with the same expert ranked by lane via match_any -- and the rank
// inside the chunk goes to src2dst, the chunk histogram to the workspace.
__device__ void endpoints_block(const int32_t* __restrict__ counts, int32_t* __restrict__ ws, int nchunks, int E,
                                int A, int32_t* __restrict__ ends, long cap, uint32_t* err, int32_t* cnt_s,
                                int32_t* warp_sums, int32_t* carry);

// The last block to finish (a completion count in the workspace, zeroed by
// the launch sequence before this kernel and again by that block) then runs
// the endpoint step over all the histograms.
__global__ void __launch_bounds__(256) rank_count_kernel(const int32_t* __restrict__ ids,
                                                         int32_t* __restrict__ s2d, int32_t* __restrict__ ws,
                                                         int T, int E, int k, int A, int32_t* __restrict__ ends,
                                                         long cap, uint32_t* err) {
  pdl_launch_dependents();  // the scatter launch may start quantising its rows now
  extern __shared__ int32_t smem_i32[];
  int32_t* cnt = smem_i32;                 // [E] running count per expert
  int32_t* ids_s = smem_i32 + E;           // [kScatterChunk * k] the chunk's expert ids
  const int c = blockIdx.x;
  const int t0 = c * kScatterChunk;
  const int t1 = min(T, t0 + kScatterChunk);
  const int nr = (t1 - t0) * k;
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  for (int r = threadIdx.x; r < nr; r += blockDim.x) ids_s[r] = ids[(size_t)t0 * k + r];
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
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
  // last block: the endpoints (histograms of every block are visible after
  // the fences around the completion count)
  __shared__ int last;
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t carry;
  unsigned int* done = reinterpret_cast<unsigned int*>(ws + (size_t)gridDim.x * E);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  endpoints_block(nullptr, ws, (int)gridDim.x, E, A, ends, cap, err, cnt, warp_sums, &carry);
  if (threadIdx.x == 0) *done = 0u;
}

// Endpoints. With `counts` given, count[e] = counts[e]; otherwise count[e] is
// the sum of the chunk histograms, which are replaced by their exclusive
// prefix over chunks (routes of e in earlier chunks). P consecutive lanes
// share an expert and split its chunks into P runs; each lane reads its run
// with independent loads, the run totals are scanned across the P lanes, and
// the run is written back. The block then scans the A-aligned counts over
// experts: start[e] = align_up(end[e-1], A), end[e] = start[e] + count[e].
// The block's work, with any block size (a multiple of 32): cnt_s [E] and
// warp_sums [32] in shared memory, carry one shared int. The histograms are
// read with ld.global.cg: in the fused launch they were written by other
// blocks of the same kernel.
__device__ void endpoints_block(const int32_t* __restrict__ counts, int32_t* __restrict__ ws, int nchunks, int E,
                                int A, int32_t* __restrict__ ends, long cap, uint32_t* err, int32_t* cnt_s,
                                int32_t* warp_sums, int32_t* carry) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (int)blockDim.x >> 5;
  if (threadIdx.x == 0) *carry = 0;
  if (counts) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt_s[e] = counts[e];
  } else {
    int P = 1;
    while (P < 32 && E * P * 2 <= (int)blockDim.x) P *= 2;
    const int sub = threadIdx.x & (P - 1);
    const int groups = blockDim.x / P;
    const int L = (nchunks + P - 1) / P;
    const int c_lo = min(nchunks, sub * L), c_hi = min(nchunks, c_lo + L);
    constexpr int U = 8;
    const int iters = (E + groups - 1) / groups;  // the same in every lane of a warp
    for (int it = 0; it < iters; ++it) {
      const int e = it * groups + (int)threadIdx.x / P;
      const bool ok = e < E;
      int tot = 0;
      if (ok) {
        for (int c0 = c_lo; c0 < c_hi; c0 += U) {
          int v[U];
#pragma unroll
          for (int u = 0; u < U; ++u) v[u] = (c0 + u < c_hi) ? __ldcg(ws + (size_t)(c0 + u) * E + e) : 0;
#pragma unroll
          for (int u = 0; u < U; ++u) tot += v[u];
        }
      }
      int incl = tot;
      for (int o = 1; o < P; o <<= 1) {
        const int n = __shfl_up_sync(kFull, incl, o, P);
        if (sub >= o) incl += n;
      }
      if (ok) {
        int run = incl - tot;
        for (int c0 = c_lo; c0 < c_hi; c0 += U) {
          int v[U];
#pragma unroll
          for (int u = 0; u < U; ++u) v[u] = (c0 + u < c_hi) ? __ldcg(ws + (size_t)(c0 + u) * E + e) : 0;
#pragma unroll
          for (int u = 0; u < U; ++u) {
            if (c0 + u < c_hi) ws[(size_t)(c0 + u) * E + e] = run;
            run += v[u];
          }
        }
        if (sub == P - 1) cnt_s[e] = incl;
      }
    }
  }
  __syncthreads();
  for (int base = 0; base < E; base += blockDim.x) {
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
      int sm = (lane < nwarps) ? warp_sums[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, sm, o);
        if (lane >= o) sm += n;
      }
      if (lane < nwarps) warp_sums[lane] = sm;
    }
    __syncthreads();
    const int start = *carry + (v - aligned) + (warp > 0 ? warp_sums[warp - 1] : 0);
    if (e < E) ends[e] = start + total;
    __syncthreads();
    if (threadIdx.x == 0) *carry += warp_sums[nwarps - 1];
    __syncthreads();
  }
  if (threadIdx.x == 0 && E > 0 && cap >= 0 && (long)ends[E - 1] > cap) raise_error(err, MOE_DEVERR_CAPACITY);
}

__global__ void __launch_bounds__(1024) endpoints_kernel(const int32_t* __restrict__ counts,
                                                         int32_t* __restrict__ ws, int nchunks, int E,
                                                         int A, int32_t* __restrict__ ends, long cap,
                                                         uint32_t* err) {
  extern __shared__ int32_t cnt_s[];  // [E]
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t carry;
  endpoints_block(counts, ws, nchunks, E, A, ends, cap, err, cnt_s, warp_sums, &carry);
}

__device__ __forceinline__ uint32_t e4m3x4(const float* f, float sc) {
  return e4m3x2_satfinite(__fmul_rn(f[0], sc), __fmul_rn(f[1], sc)) |
         (e4m3x2_satfinite(__fmul_rn(f[2], sc), __fmul_rn(f[3], sc)) << 16);
}

// One warp per token, in two phases. Before griddepcontrol.wait, which
// returns once the rank/count launch has completed (the kernel is launched to
// start while that launch still runs): the token row is quantised once (16
// lanes per 128-column group, or 4 per 32-column group in the MXFP8 recipe;
// uint4 loads, four in flight per lane) into the warp's shared-memory stash,
// codes then scale bytes. After it: the final src2dst of each slot and the
// copies of the stash to every destination row (16-byte stores) and of the
// scale bytes, as packed words, to every destination's column of a_sf.
__global__ void __launch_bounds__(256) scatter_quant_kernel(const uint16_t* __restrict__ x,
                                                            const int32_t* __restrict__ ids,
                                                            int32_t* __restrict__ s2d,
                                                            const int32_t* __restrict__ ws,
                                                            const int32_t* __restrict__ ends,
                                                            uint8_t* __restrict__ a_fp8,
                                                            int32_t* __restrict__ a_sf, int T, int E,
                                                            int k, int A, int H, int ld_sf, long cap,
                                                            bool g32, uint32_t* err) {
  extern __shared__ __align__(16) uint8_t stash_all[];
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int nsb = g32 ? H / 32 : H / 128;  // scale bytes of a row
  const int nwords = (nsb + 3) / 4;         // packed scale words of a row
  const int stride = H + (nsb + 15) / 16 * 16;
  uint8_t* stash = stash_all + (size_t)(threadIdx.x >> 5) * stride;
  const int npass = (H + 255) / 256;
  bool waited = false;
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += gridDim.x * wpb) {
    const uint16_t* xr = x + (size_t)t * H;
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
        // 16 lanes per 128-column group, or 4 per 32-column group (MXFP8)
        for (int o = g32 ? 2 : 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
        const uint32_t b = active ? group_scale_byte(amax) : 0u;
        const float sc = pow2_f32(127 - (int)b);
        if (active) {
          uint2 codes;
          codes.x = e4m3x4(f, sc);
          codes.y = e4m3x4(f + 4, sc);
          *reinterpret_cast<uint2*>(stash + col) = codes;
          if ((lane & (g32 ? 3 : 15)) == 0) stash[H + (g32 ? col / 32 : col / 128)] = (uint8_t)b;
        }
      }
    }
    __syncwarp();
    if (!waited) {
      pdl_wait();  // src2dst ranks, chunk prefixes and endpoints are complete from here on
      waited = true;
    }
    int dst = -1;
    if (lane < k) {
      const int e = ids[(size_t)t * k + lane];
      const int lr = s2d[(size_t)t * k + lane];
      if (e >= 0 && e < E && lr >= 0) {
        const int start = (e == 0) ? 0 : (int)align_up64(ends[e - 1], A);
        dst = start + ws[(size_t)(t / kScatterChunk) * E + e] + lr;
        if ((long)dst >= cap) {
          raise_error(err, MOE_DEVERR_CAPACITY);
          dst = -1;
        }
      }
      s2d[(size_t)t * k + lane] = dst;
    }
    // codes: 16 bytes per lane per step, four steps in registers, stored to every destination
    const int n16 = H / 16;
    for (int c0 = 0; c0 < n16; c0 += 128) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + 32 * u + lane;
        if (c < n16) v[u] = *reinterpret_cast<const uint4*>(stash + 16 * c);
      }
      for (int j = 0; j < k; ++j) {
        const int d = __shfl_sync(kFull, dst, j);
        if (d < 0) continue;
        uint8_t* row = a_fp8 + (size_t)d * H;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = c0 + 32 * u + lane;
          if (c < n16) *reinterpret_cast<uint4*>(row + 16 * c) = v[u];
        }
      }
    }
    // scale words: byte (g % 4) of word g / 4, unused bytes of the last word 0
    for (int w0 = 0; w0 < nwords; w0 += 32) {
      const int w = w0 + lane;
      uint32_t word = 0;
      if (w < nwords)
        for (int i = 0; i < 4; ++i)
          if (4 * w + i < nsb) word |= (uint32_t)stash[H + 4 * w + i] << (8 * i);
      for (int j = 0; j < k; ++j) {
        const int d = __shfl_sync(kFull, dst, j);
        if (d >= 0 && w < nwords) a_sf[(size_t)w * ld_sf + d] = (int32_t)word;
      }
    }
    __syncwarp();  // the stash is refilled by the warp's next token
  }
}

template <int EPL, int MODE>
cudaError_t launch_route(const moe_route_args& a, int num_sms, unsigned int* done, cudaStream_t st) {
  const int blocks = (int)lmin((a.T + 7) / 8, (long)num_sms * 8);
  route_kernel<EPL, MODE><<<blocks, 256, 0, st>>>(a.logits, a.corr_bias, a.topk_ids, a.topk_w, a.T, a.E, a.k,
                                                  done);
  return cudaGetLastError();
}

template <int MODE>
cudaError_t dispatch_epl(const moe_route_args& a, int num_sms, unsigned int* done, cudaStream_t st) {
  const int epl = (a.E + 31) / 32;
  if (epl <= 1) return launch_route<1, MODE>(a, num_sms, done, st);
  if (epl <= 2) return launch_route<2, MODE>(a, num_sms, done, st);
  if (epl <= 4) return launch_route<4, MODE>(a, num_sms, done, st);
  if (epl <= 8) return launch_route<8, MODE>(a, num_sms, done, st);
  if (epl <= 16) return launch_route<16, MODE>(a, num_sms, done, st);
  if (epl <= 24) return launch_route<24, MODE>(a, num_sms, done, st);
  return launch_route<32, MODE>(a, num_sms, done, st);
}

}  // namespace

// Shared memory of a scatter block: eight warps' stashes of a quantised row
// (H codes, then the scale bytes rounded up to 16).
size_t scatter_stash_bytes(int H, bool g32) {
  const int nsb = g32 ? H / 32 : H / 128;
  return (size_t)8 * (size_t)(H + (nsb + 15) / 16 * 16);
}

cudaError_t init_route_scatter() {
  return cudaFuncSetAttribute(scatter_quant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kScatterStashMax);
}

// Chunk histograms [nchunks][E] int32, then the 4-byte completion count of
// the rank/count launch, rounded up to 16 bytes.
size_t route_scatter_ws_bytes(int T, int E, int k) {
  (void)k;
  const size_t nchunks = (size_t)(T + kScatterChunk - 1) / kScatterChunk;
  const size_t b = nchunks * (size_t)E * sizeof(int32_t) + sizeof(uint32_t);
  return (b + 15) / 16 * 16;
}

cudaError_t launch_expert_ends(const int32_t* counts, int E, int A, int32_t* ends, uint32_t* err,
                               cudaStream_t st) {
  endpoints_kernel<<<1, 1024, (size_t)E * sizeof(int32_t), st>>>(counts, nullptr, 0, E, A, ends, -1, err);
  return cudaGetLastError();
}

cudaError_t launch_route_scatter(const moe_route_args& a, int num_sms, uint32_t* err, cudaStream_t st) {
  const int nchunks = (a.T + kScatterChunk - 1) / kScatterChunk;
  cudaError_t ce = cudaSuccess;
  int32_t* ws = (int32_t*)a.workspace;
  if (a.T > 0) {
    // completion count of rank_count_kernel, zeroed by the routing kernel
    // (or a 4-byte memset when the routing is given)
    unsigned int* done = reinterpret_cast<unsigned int*>(ws + (size_t)nchunks * a.E);
    if (a.routing_mode == MOE_ROUTE_SOFTMAX_TOPK)
      ce = dispatch_epl<MOE_ROUTE_SOFTMAX_TOPK>(a, num_sms, done, st);
    else if (a.routing_mode == MOE_ROUTE_SIGMOID_BIAS_TOPK)
      ce = dispatch_epl<MOE_ROUTE_SIGMOID_BIAS_TOPK>(a, num_sms, done, st);
    else
      ce = cudaMemsetAsync(done, 0, sizeof(unsigned int), st);
    if (ce != cudaSuccess) return ce;
    const size_t smem = (size_t)(a.E + kScatterChunk * a.k) * sizeof(int32_t);
    rank_count_kernel<<<nchunks, 256, smem, st>>>(a.topk_ids, a.src2dst, ws, a.T, a.E, a.k, a.A, a.expert_ends,
                                                  a.cap, err);
    if ((ce = cudaGetLastError()) != cudaSuccess) return ce;
    const int blocks = (int)lmin((a.T + 7) / 8, (long)num_sms * 16);
    return launch_maybe_pdl(scatter_quant_kernel, dim3(blocks), dim3(256), scatter_stash_bytes(a.H, a.quant_group == 32),
                            st, true, a.x, (const int32_t*)a.topk_ids, a.src2dst, (const int32_t*)ws,
                            (const int32_t*)a.expert_ends, a.a_fp8, a.a_sf, a.T, a.E, a.k, a.A, a.H,
                            (int)align_up64(a.cap, 4), (long)a.cap, a.quant_group == 32, err);
  }
  // no tokens: every expert is empty
  endpoints_kernel<<<1, 1024, (size_t)a.E * sizeof(int32_t), st>>>(nullptr, ws, 0, a.E, a.A, a.expert_ends, a.cap,
                                                                   err);
  return cudaGetLastError();
}

// ---------------------------------------------------- no-allocation variant
// Scratch of moe_route_scatter_noalloc: the per-chunk expert histograms (up
// to 1 MiB) and the rank/count completion count live in this file-scope
// device array instead of a caller-provided workspace. Every GPU that loads
// this module holds these 1 MiB + 16 bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = (size_t(1) << 20) + 16;
static __device__ __align__(256) int32_t g_route_scratch[kNoAllocScratchBytes / sizeof(int32_t)];

size_t route_scatter_noalloc_max_bytes() { return kNoAllocScratchBytes; }

// Device address of the scratch array on the current device. In host code
// the array's name is only a stand-in, never a device address; the address
// comes from the runtime. Looking it up also loads this module on the device
// (with lazy loading the array is created then). Called once per context, at
// its creation, with the context's device current.
cudaError_t route_scatter_noalloc_scratch(void** addr) {
  *addr = nullptr;
  return cudaGetSymbolAddress(addr, g_route_scratch);
}

// `scratch` is the address route_scatter_noalloc_scratch returned for the
// current device.
cudaError_t launch_route_scatter_noalloc(const moe_route_args& a, void* scratch, int num_sms, uint32_t* err,
                                         cudaStream_t st) {
  if (!scratch) return cudaErrorInvalidDevicePointer;
  moe_route_args b = a;
  b.workspace = scratch;
  b.workspace_bytes = kNoAllocScratchBytes;
  return launch_route_scatter(b, num_sms, err, st);
}

}  // namespace moe
