// combine.cu -- top-k weighted combine and load-time weight preparation.
//
// Combine ([DG] §2.6.1, post_reorder): out[t] = bf16(rsf * sum_j w[t,j] *
// down[src2dst[t,j]]) over the slots with src2dst >= 0, fp32 accumulation,
// one fused multiply-add per slot in slot order. A warp per work item (token,
// 256 columns), 8 columns per lane: lanes j < k hold the token's slot j
// (src2dst, weight), broadcast by shuffles; uint4 gathers from the k grouped
// rows, a uint4 store. The slot data of the warp's next item is loaded while
// the current item's gathers are in flight, so an item costs one memory
// round trip instead of two dependent ones. k > 32 takes
// combine_kernel_wide, a thread per (token, 8 columns).
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr unsigned kFullMask = 0xFFFFFFFFu;
// Grid: one wave of resident blocks (80 registers per thread: 3 blocks of 256
// threads per SM; 2 or 4 measured slower).
constexpr int kCombineBlocksPerSm = 3;

__global__ void __launch_bounds__(256, kCombineBlocksPerSm) combine_kernel(const uint16_t* __restrict__ down, int H,
                                                      const float* __restrict__ topk_w,
                                                      const int32_t* __restrict__ s2d, int T, int k,
                                                      float rsf, uint16_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int cb = (H + 255) / 256;  // 256-column blocks per token
  const long n_items = (long)T * cb;
  const long wstride = (long)gridDim.x * (blockDim.x / 32);
  long item = (long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  int nxt_dst = -1;
  float nxt_w = 0.0f;
  auto load_slots = [&](long it) {
    nxt_dst = -1;
    nxt_w = 0.0f;
    if (it < n_items && lane < k) {
      const size_t o = (size_t)(it / cb) * k + lane;
      nxt_dst = s2d[o];
      nxt_w = topk_w[o];
    }
  };
  load_slots(item);
  for (; item < n_items; item += wstride) {
    const int my_dst = nxt_dst;
    const float my_w = nxt_w;
    load_slots(item + wstride);
    const int t = (int)(item / cb);
    const int c = (int)(item % cb) * 256 + lane * 8;
    const bool in = c < H;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int j0 = 0; j0 < k; j0 += 8) {
      int dst[8];
      float wt[8];
      uint4 v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        dst[q] = __shfl_sync(kFullMask, my_dst, (j0 + q) & 31);
        wt[q] = __shfl_sync(kFullMask, my_w, (j0 + q) & 31);
        if (j0 + q >= k) dst[q] = -1;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q)
        v[q] = (dst[q] >= 0 && in) ? __ldg(reinterpret_cast<const uint4*>(down + (size_t)dst[q] * H + c))
                                   : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (dst[q] < 0) continue;
        const uint32_t* pv = &v[q].x;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] = __fmaf_rn(wt[q], bf16_lo(pv[i]), acc[2 * i]);
          acc[2 * i + 1] = __fmaf_rn(wt[q], bf16_hi(pv[i]), acc[2 * i + 1]);
        }
      }
    }
    if (in) {
      uint4 o;
      uint32_t* po = &o.x;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        po[i] = pack_bf16x2(__fmul_rn(acc[2 * i], rsf), __fmul_rn(acc[2 * i + 1], rsf));
      *reinterpret_cast<uint4*>(out + (size_t)t * H + c) = o;
    }
  }
}

__global__ void __launch_bounds__(256) combine_kernel_wide(const uint16_t* __restrict__ down, int H,
                                                      const float* __restrict__ topk_w,
                                                      const int32_t* __restrict__ s2d, int T, int k,
                                                      float rsf, uint16_t* __restrict__ out) {
  const int chunks = H / 8;
  const long total = (long)T * chunks;
  for (long idx = (long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long)gridDim.x * blockDim.x) {
    const int t = (int)(idx / chunks);
    const int c = (int)(idx % chunks);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int j0 = 0; j0 < k; j0 += 8) {
      int dst[8];
      float wt[8];
      uint4 v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int j = j0 + q;
        dst[q] = (j < k) ? s2d[(size_t)t * k + j] : -1;
        wt[q] = (j < k) ? topk_w[(size_t)t * k + j] : 0.0f;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q)
        v[q] = (dst[q] >= 0) ? __ldg(reinterpret_cast<const uint4*>(down + (size_t)dst[q] * H) + c)
                             : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (dst[q] < 0) continue;
        const uint32_t* pv = &v[q].x;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] = __fmaf_rn(wt[q], bf16_lo(pv[i]), acc[2 * i]);
          acc[2 * i + 1] = __fmaf_rn(wt[q], bf16_hi(pv[i]), acc[2 * i + 1]);
        }
      }
    }
    uint4 o;
    uint32_t* po = &o.x;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      po[i] = pack_bf16x2(__fmul_rn(acc[2 * i], rsf), __fmul_rn(acc[2 * i + 1], rsf));
    reinterpret_cast<uint4*>(out + (size_t)t * H)[c] = o;
  }
}

// Scales [E][N][K/32] bytes -> words [E][K/128][N]: the word of (e, c, n)
// holds the four bytes sf[e][n][4c .. 4c+3], byte 4c lowest; inside every
// block of 128 rows, position 4 i + j holds row 32 j + i (the source layout of
// tcgen05.cp 32x128b.warpx4, so the GEMM copies it without rearranging).
// Source row of output row n: identity, or (gate/up interleave in blocks of
// 128) output rows 256b .. 256b+127 take gate rows 128b .., rows 256b+128 ..
// take up rows N/2 + 128b ...
__device__ __forceinline__ int src_row(int n, int N, bool blocked) {
  if (!blocked) return n;
  const int b = n >> 8, w = n & 255;
  return (w < 128) ? (b << 7) + w : (N >> 1) + (b << 7) + (w - 128);
}

// sf_block: the input holds one scale per 128 x 128 weight block,
// [E][ceil(N/128)][K/128] (FP8 block128 recipe); each of the block's
// 32-K scale slots takes it.
__global__ void prepare_scales_kernel(const uint8_t* __restrict__ sf_in, int E, int N, int K, bool blocked,
                                      bool sf_block, uint32_t* __restrict__ sf_out) {
  const int KC = K / 128;
  const long total = (long)E * KC * N;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
    const int pos = (int)(i % N);
    const int q = pos & 127;
    const int n = (pos & ~127) + 32 * (q & 3) + (q >> 2);
    const long ec = i / N;
    const int c = (int)(ec % KC);
    const int e = (int)(ec / KC);
    if (sf_block) {
      const uint32_t b = sf_in[((size_t)e * ((N + 127) / 128) + src_row(n, N, blocked) / 128) * KC + c];
      sf_out[i] = b * 0x01010101u;
    } else {
      const uint8_t* p = sf_in + ((size_t)e * N + src_row(n, N, blocked)) * (K / 32) + 4 * c;
      sf_out[i] = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
    }
  }
}

// Packed e2m1 byte pairs -> e4m3 codes (exact: every e2m1 value is an e4m3
// value), or a copy; rows remapped by src_row. One thread per output byte
// pair (e4m3) or byte (a copy of e2m1, or of e4m3 input when in8).
__global__ void weights_kernel(const uint8_t* __restrict__ w_in, int E, int N, int K, bool blocked, bool widen,
                               bool in8, uint8_t* __restrict__ w_out) {
  const long rowb = in8 ? K : K / 2;
  const long nbytes = (long)E * N * rowb;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < nbytes; i += (long)gridDim.x * blockDim.x) {
    const long rowi = i / rowb, col = i % rowb;
    const int e = (int)(rowi / N), n = (int)(rowi % N);
    const uint32_t b = w_in[((long)e * N + src_row(n, N, blocked)) * rowb + col];
    if (widen) {
      const float lo = e2m1_to_f32(b & 0xFu), hi = e2m1_to_f32(b >> 4);
      reinterpret_cast<uint16_t*>(w_out)[i] = (uint16_t)e4m3x2_satfinite(lo, hi);
    } else {
      w_out[i] = (uint8_t)b;
    }
  }
}

}  // namespace

cudaError_t launch_combine(const uint16_t* down, int H, const float* topk_w, const int32_t* src2dst,
                           int T, int k, float rsf, uint16_t* out, int num_sms, cudaStream_t st) {
  const long total = (long)T * (H / 8);
  if (total == 0) return cudaSuccess;
  if (k > 32) {
    const int blocks = (int)lmin((total + 255) / 256, (long)num_sms * 8);
    combine_kernel_wide<<<blocks, 256, 0, st>>>(down, H, topk_w, src2dst, T, k, rsf, out);
    return cudaGetLastError();
  }
  const long items = (long)T * ((H + 255) / 256);
  const int blocks = (int)lmin((items + 7) / 8, (long)num_sms * kCombineBlocksPerSm);
  combine_kernel<<<blocks, 256, 0, st>>>(down, H, topk_w, src2dst, T, k, rsf, out);
  return cudaGetLastError();
}

cudaError_t launch_prepare_weights(const uint8_t* w_in, const uint8_t* sf_in, int E, int N, int K,
                                   int w_format, uint8_t* w_out, uint32_t* sf_out, cudaStream_t st) {
  const bool blocked = (w_format & MOE_GEMM_W_GATEUP_BLOCK128) != 0;
  const bool in8 = (w_format & MOE_GEMM_W_IN_E4M3) != 0;
  const bool widen = (w_format & MOE_GEMM_W_E4M3) != 0 && !in8;
  const bool sf_block = (w_format & MOE_GEMM_W_SF_BLOCK128) != 0;
  const long words = (long)E * (K / 128) * N;
  if (words > 0) {
    prepare_scales_kernel<<<(int)lmin((words + 255) / 256, 65535), 256, 0, st>>>(sf_in, E, N, K, blocked, sf_block,
                                                                                 sf_out);
    cudaError_t ce = cudaGetLastError();
    if (ce != cudaSuccess) return ce;
  }
  const long nbytes = (long)E * N * (in8 ? K : K / 2);
  if (nbytes == 0) return cudaSuccess;
  if (!blocked && !widen) {
    if (w_out != w_in) return cudaMemcpyAsync(w_out, w_in, (size_t)nbytes, cudaMemcpyDeviceToDevice, st);
    return cudaSuccess;
  }
  weights_kernel<<<(int)lmin((nbytes + 255) / 256, 65535), 256, 0, st>>>(w_in, E, N, K, blocked, widen, in8,
                                                                          w_out);
  return cudaGetLastError();
}

}  // namespace moe
