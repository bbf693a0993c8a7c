// decode_gemm.cu -- the small-batch decode path on the tcgen05 tensor cores
// (up to 128 tokens): every selected local expert's weights are read once and
// multiplied against all the token slots that chose it.
//
// [SD] §3 computes, per (token, slot) whose expert is local, two GEMVs with a
// GLU between them and a weighted sum over the slots; [SD] §4 keeps that path
// to num_tokens <= 8 because each token re-reads its experts' weights. With
// the slots grouped by expert nothing is re-read, so the same computation runs
// here for any batch up to 128 tokens as four launches:
//
//   decode_split_kernel       slots grouped by local expert into segments with
//                             16-row aligned starts ([LR] §2 endpoint layout,
//                             A = 16); each slot's x row split into two e4m3
//                             terms with group-32 UE8M0 scales
//   decode_gemm_kernel<GLU>   y1 = W_gu x (* scale) + b, act = GLU(y1), and
//                             act split the same way for the next GEMM
//   decode_gemm_kernel        y2 = W_d act (* scale) + b
//   weighted_sum_kernel       (decode.cu) out = slot-ordered sum of topk_w y2
//
// Operands of tcgen05.mma.kind::mxf8f6f4.block_scale (M128, N256, K32): the
// weights are the B operand, 256 rows per tile (with the GLU the gate and the
// up 128-row blocks of the same output rows), moved by TMA in their stored
// format (e4m3, or e2m1 expanded to a byte per element by the 16U4_ALIGN16B
// tensor-map type) with their UE8M0 group-32 scales -- FP8-per-expert weights
// take unit scales and their fp32 scale in the epilogue; the A operand holds
// the two activation terms of up to 32 slots (64 rows; the accumulator lanes
// of the other 64 rows are never read). A small-N MMA costs about as much as
// a wide one, so the wide side goes to the weights: 4 MMAs per 128-wide K
// block.
//
// Two-term activation split. For a group of 32 bf16 values v with absolute
// maximum a:
//   hi = e4m3(v 2^(127-sh)), sh = UE8M0 scale byte of a / 448,
//   r  = v - hi 2^(sh-127)            (exact in fp32),
//   lo = e4m3(r 2^(127-sl)), sl = the scale byte of max|r| / 448,
// and the MMA accumulates W hi 2^(sh-127) + W lo 2^(sl-127) in fp32 tensor
// memory. bf16 carries 8 significant bits and each e4m3 term 4, so hi + lo is
// v exactly for every value within 2^13 of its group's maximum; smaller
// values keep an absolute error below 2^-21 of that maximum.
//
// GEMM kernel structure (one persistent CTA per SM, 256 threads), as in the
// grouped GEMM of the layer path:
//   warp 0    producer: the tile's weight scale rows (MXFP4, one bulk copy per
//             tile), then per 128-wide K block the activation terms' scale
//             words (bulk), the A tile (activation terms) and the B tile
//             (weights; the gate and up blocks with GLU) by TMA
//   warp 1    TMEM owner and MMA issuer: one 128 x 256 fp32 accumulator,
//             released by the epilogue once it has read it
//   warp 2    scale transposer: A and B scale words into the 32-row x 16-byte
//             source layout of tcgen05.cp 32x128b.warpx4
//   warps 4-7 epilogue: tcgen05.ld, bias, GLU and the split of act, or bias
//             only; one thread per weight row, one column per slot
// Tiles are (local expert, 128 output rows, chunk of <= 64 slots), in expert
// order with the chunks of one row block adjacent, so a weight block that
// serves two chunks is read from HBM once and from L2 once.
// Every mbarrier wait is bounded; a wait that runs out sets
// MOE_DEVERR_WAIT_TIMEOUT and every role leaves its loop.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "pipeline.cuh"
#include "tcgen05.cuh"

namespace moe {

namespace {

constexpr unsigned kAll = 0xFFFFFFFFu;
constexpr int kDgThreads = 256;
constexpr int kDgChunk = 32;  // slots per tile (A tile: 64 rows of activation terms)
constexpr int kDgAlign = 16;  // segment starts and the MMA's N granularity
constexpr int kDgMaxLocal = 1024;
constexpr int kDgMaxSlots = 4096;
constexpr int kDgMaxKs = 128;  // MXFP4 scale bytes per weight row (K <= 4096)
constexpr int kEpiStride = 257;  // floats per staged slot row: 128 gate + 128 up + 1 (bank spread)
constexpr int kEpiSlots = 8;     // slots staged per GLU epilogue pass
constexpr int kMaxStages = 6;
constexpr int kDgBK = 128;

// Stage layout (bytes): the 64 x 128 A tile (activation terms of up to 32
// slots; the MMA's M = 128 also reads the next 64 rows, whose accumulator
// lanes are never used), the 256 x 128 B tile (two 128-row weight blocks), the
// tcgen05.cp sources of the A and B scales, and the A scale words as copied
// (64, in split-row order).
constexpr uint32_t kStA = 0, kStB = 8192;
constexpr uint32_t kStSfa = 40960;
constexpr uint32_t kStSfb = 41472;   // + 512 * block
constexpr uint32_t kStSfin = 42496;
constexpr uint32_t kStBytes = 43008;  // 42 KB, keeps every stage 1024-byte aligned
constexpr uint32_t kSmemMax = 232448;

// Shared-memory layout, computed on the host from the weight format and K: as
// many stages as fit (the bytes in flight per SM set the streaming rate), the
// MXFP4 tile scale rows (two buffers of 256 rows x K/32 bytes), the GLU
// staging rows, the tile prefix, the barriers.
struct DgLayout {
  int stages;
  uint32_t tsf, tsf_bytes, epi, prefix, bar, tmem_slot, abort_flag, scan, bytes;
};

DgLayout dg_layout(bool fp4, int Ks) {
  DgLayout L{};
  L.tsf_bytes = fp4 ? (uint32_t)(256 * Ks + 15) / 16 * 16 : 0u;
  const uint32_t epi_bytes = kEpiSlots * kEpiStride * 4 + 16;
  const uint32_t prefix_bytes = (kDgMaxLocal + 1) * 4 + 4;
  const uint32_t tail = epi_bytes + prefix_bytes + (3 * kMaxStages + 7) * 8 + 4 + 4 + 32 * 4;
  const uint32_t fixed = 2 * L.tsf_bytes + tail + 1024;  // + slack for the 1024-byte alignment
  L.stages = (int)((kSmemMax - fixed) / kStBytes);
  if (L.stages > kMaxStages) L.stages = kMaxStages;
  L.tsf = (uint32_t)L.stages * kStBytes;
  L.epi = L.tsf + 2 * L.tsf_bytes;
  L.prefix = L.epi + epi_bytes;
  L.bar = L.prefix + prefix_bytes;  // 8-byte aligned: every term above is a multiple of 8
  L.tmem_slot = L.bar + (3 * L.stages + 7) * 8;
  L.abort_flag = L.tmem_slot + 4;
  L.scan = L.abort_flag + 4;
  L.bytes = L.scan + 32 * 4 + 1024;
  return L;
}

__host__ __device__ constexpr int align16i(int v) { return (v + kDgAlign - 1) / kDgAlign * kDgAlign; }

// Split row of term h (0 hi, 1 lo) of segment row r: blocks of 16 segment rows
// become 16 hi rows followed by 16 lo rows, so that in the MMA's accumulator
// the two terms of a slot sit in lanes j and j + 16 of one warp.
__host__ __device__ __forceinline__ int split_row(int r, int h) { return 32 * (r >> 4) + 16 * h + (r & 15); }

// Exclusive prefix over v(0..n-1) by the whole block (n <= 4 * blockDim.x):
// out[e] = v(0) + ... + v(e-1), out[n] = the total. Ends with a barrier.
template <typename F>
__device__ void block_exclusive_scan(int n, F v, int32_t* out, int32_t* tmp) {
  const int per = (n + (int)blockDim.x - 1) / (int)blockDim.x;
  const int lo = min(n, (int)threadIdx.x * per), hi = min(n, lo + per);
  int sum = 0;
  for (int e = lo; e < hi; ++e) sum += v(e);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kAll, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) tmp[warp] = incl;
  __syncthreads();
  int run = incl - sum;
  for (int w = 0; w < warp; ++w) run += tmp[w];
  for (int e = lo; e < hi; ++e) {
    out[e] = run;
    run += v(e);
  }
  if (threadIdx.x == blockDim.x - 1) out[n] = run;
  __syncthreads();
}

// Two-term split of four values of one group held by a lane, the group's 32
// values spread over 8 consecutive lanes (collective over the warp; each
// 8-lane group reduces its own maximum): the four hi and lo codes packed as
// bytes, and the group's scale bytes.
__device__ __forceinline__ void split_quad(const float (&v)[4], uint32_t& hq, uint32_t& lq, uint32_t& sh,
                                           uint32_t& sl) {
  float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(kAll, m, o));
  sh = group_scale_byte(m);
  const float up_h = pow2_f32(127 - (int)sh), down_h = pow2_f32((int)sh - 127);
  const uint32_t h01 = e4m3x2_satfinite(__fmul_rn(v[0], up_h), __fmul_rn(v[1], up_h));
  const uint32_t h23 = e4m3x2_satfinite(__fmul_rn(v[2], up_h), __fmul_rn(v[3], up_h));
  const float2 d01 = e4m3x2_to_f32x2(h01), d23 = e4m3x2_to_f32x2(h23);
  float r[4];
  r[0] = __fsub_rn(v[0], __fmul_rn(d01.x, down_h));
  r[1] = __fsub_rn(v[1], __fmul_rn(d01.y, down_h));
  r[2] = __fsub_rn(v[2], __fmul_rn(d23.x, down_h));
  r[3] = __fsub_rn(v[3], __fmul_rn(d23.y, down_h));
  float mr = fmaxf(fmaxf(fabsf(r[0]), fabsf(r[1])), fmaxf(fabsf(r[2]), fabsf(r[3])));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) mr = fmaxf(mr, __shfl_xor_sync(kAll, mr, o));
  sl = group_scale_byte(mr);
  const float up_l = pow2_f32(127 - (int)sl);
  hq = (h01 & 0xFFFFu) | (h23 << 16);
  lq = (e4m3x2_satfinite(__fmul_rn(r[0], up_l), __fmul_rn(r[1], up_l)) & 0xFFFFu) |
       (e4m3x2_satfinite(__fmul_rn(r[2], up_l), __fmul_rn(r[3], up_l)) << 16);
}

struct DsArgs {
  const int32_t* ids;
  int T, k, expert_start, n_local;
  const uint16_t* x;  // [T][H]
  int H;
  int32_t* cnt;       // [n_local]
  int32_t* seg;       // [n_local]
  int32_t* row_slot;  // [R]
  uint8_t* xs;        // [2R][H] split rows
  uint32_t* xsf;      // [ceil(H/128)][2R]
  int R;
};

// Segments and the split of x. Every CTA derives the same counts, segment
// starts and per-slot ranks from topk_ids (the rank of a slot is the number
// of earlier slots with the same expert, so the order is deterministic); CTA
// 0 writes the counts, the starts and the padding entries of row_slot. Work
// items are (slot, 128-element block): a warp loads the block (8 bytes per
// lane; lanes 8b..8b+7 hold group b), splits it and writes 128 hi and 128 lo
// codes and the block's two scale words.
__global__ void __launch_bounds__(256) decode_split_kernel(const __grid_constant__ DsArgs a) {
  __shared__ int32_t cnt_s[kDgMaxLocal];
  __shared__ int32_t seg_s[kDgMaxLocal + 1];
  __shared__ int32_t lid_s[kDgMaxSlots];
  __shared__ int32_t tmp[32];
  const int S = a.T * a.k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < a.n_local; e += blockDim.x) cnt_s[e] = 0;
  __syncthreads();
  for (int s = threadIdx.x; s < S; s += blockDim.x) {
    const int id = a.ids[s];
    const int lid = (id >= a.expert_start && id - a.expert_start < a.n_local) ? id - a.expert_start : -1;
    lid_s[s] = lid;
    if (lid >= 0) atomicAdd(&cnt_s[lid], 1);
  }
  __syncthreads();
  block_exclusive_scan(a.n_local, [&](int e) { return align16i(cnt_s[e]); }, seg_s, tmp);
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e < a.n_local; e += blockDim.x) {
      a.cnt[e] = cnt_s[e];
      a.seg[e] = seg_s[e];
      for (int r = seg_s[e] + cnt_s[e]; r < seg_s[e + 1]; ++r) a.row_slot[r] = -1;
    }
    for (int r = seg_s[a.n_local] + (int)threadIdx.x; r < a.R; r += blockDim.x) a.row_slot[r] = -1;
  }
  const int H = a.H, W = (H + kDgBK - 1) / kDgBK;
  const long items = (long)S * W;
  for (long it = (long)blockIdx.x * 8 + warp; it < items; it += (long)gridDim.x * 8) {
    const int s = (int)(it / W), w = (int)(it % W);
    const int lid = lid_s[s];
    if (lid < 0) continue;  // warp-uniform
    const int col = kDgBK * w + 4 * lane;  // first of this lane's four elements
    const bool in = col < H;               // H % 32 == 0: whole groups in or out
    uint2 p = make_uint2(0u, 0u);
    if (in) p = __ldg(reinterpret_cast<const uint2*>(a.x + (size_t)(s / a.k) * H + col));
    int c = 0;
    for (int s2 = lane; s2 < s; s2 += 32) c += (lid_s[s2] == lid);
    const int row = seg_s[lid] + __reduce_add_sync(kAll, c);
    if (w == 0 && lane == 0) a.row_slot[row] = s;
    const float v[4] = {bf16_lo(p.x), bf16_hi(p.x), bf16_lo(p.y), bf16_hi(p.y)};
    uint32_t hq, lq, sh, sl;
    split_quad(v, hq, lq, sh, sl);
    const int rh = split_row(row, 0), rl = split_row(row, 1);
    if (in) {
      *reinterpret_cast<uint32_t*>(a.xs + (size_t)rh * H + col) = hq;
      *reinterpret_cast<uint32_t*>(a.xs + (size_t)rl * H + col) = lq;
    }
    // scale words: byte b from lane 8b; groups past H keep unit scales
    uint32_t wh = 0, wl = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t bh = __shfl_sync(kAll, in ? sh : 0x7Fu, 8 * b);
      const uint32_t bl = __shfl_sync(kAll, in ? sl : 0x7Fu, 8 * b);
      wh |= bh << (8 * b);
      wl |= bl << (8 * b);
    }
    if (lane == 0) {
      a.xsf[(size_t)w * 2 * a.R + rh] = wh;
      a.xsf[(size_t)w * 2 * a.R + rl] = wl;
    }
  }
}

struct DgArgs {
  const int32_t* cnt;       // [n_local] slots per local expert
  const int32_t* seg;       // [n_local] first segment row of the expert
  const int32_t* row_slot;  // [R] slot t*k+j of each segment row, -1 for padding
  int n_local, R;
  const uint32_t* asf;  // [KC][2R] scale words of the activation terms (split rows)
  const uint8_t* wsf;   // MXFP4: [n_local][rows][K/32]
  const float* wscale;  // FP8: [n_local]
  const uint16_t* bias;  // [n_local][rows]
  int K, M, rows;        // reduction length; output rows (I with GLU, else H); weight rows per expert
  int interleaved;
  float alpha, beta, limit;
  uint16_t* y;        // [T*k][rows]
  uint16_t* act;      // GLU: [T*k][M]
  uint8_t* a_split;   // GLU: [2R][M] e4m3 terms of act (split rows)
  uint32_t* a_sf;     // GLU: [ceil(M/128)][2R]
  uint32_t* err;
  DgLayout lay;
};

// Instruction descriptor: A (activation terms) e4m3, B (weights) e2m1 (5) or
// e4m3 (0), both K-major, N = 256 (N >> 3 at bit 17), UE8M0 scales (bit 23),
// M = 128 (M >> 4 at bit 24); the scale-factor ids (B at bit 4, A at bit 29)
// are or-ed in per K32 step.
__host__ __device__ constexpr uint32_t dg_idesc(bool b_fp4) {
  return ((b_fp4 ? 5u : 0u) << 10) | ((uint32_t)(256 >> 3) << 17) | (1u << 23) | ((uint32_t)(128 >> 4) << 24);
}

template <bool kFp4, bool kGlu>
__global__ void __launch_bounds__(kDgThreads, 1) decode_gemm_kernel(const __grid_constant__ CUtensorMap tmW,
                                                                    const __grid_constant__ CUtensorMap tmWt,
                                                                    const __grid_constant__ CUtensorMap tmA,
                                                                    const __grid_constant__ DgArgs a) {
  const DgLayout& L = a.lay;
  const int S = L.stages;
  constexpr int RT = kGlu ? 128 : 256;  // output rows per tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_flag);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.tmem_slot);
  int32_t* P = reinterpret_cast<int32_t*>(smem + L.prefix);
  const uint32_t bar0 = sbase + L.bar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto sfin_bar = [&](int s) { return bar0 + 8u * (2 * S + s); };
  auto tsf_full = [&](int b) { return bar0 + 8u * (3 * S + b); };
  auto tsf_empty = [&](int b) { return bar0 + 8u * (3 * S + 2 + b); };
  const uint32_t acc_full = bar0 + 8u * (3 * S + 4);
  const uint32_t acc_empty = bar0 + 8u * (3 * S + 5);
  const uint32_t done_bar = bar0 + 8u * (3 * S + 6);
  auto stage = [&](int s) { return smem + (size_t)s * kStBytes; };

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 2);   // producer's expect_tx arrive + transposer's arrive
      mbar_init(empty_bar(s), 1);  // tcgen05.commit
      mbar_init(sfin_bar(s), 1);   // producer's expect_tx arrive for the activation scale words
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tsf_full(b), 1);
      mbar_init(tsf_empty(b), 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kGlu ? 1 : 4);  // GLU: the warp that reads last; else one arrive per epilogue warp
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // The segments, the activation terms and their scales come from the
  // preceding kernels of the stream.
  pdl_wait();
  const int nmb = (a.M + RT - 1) / RT;
  block_exclusive_scan(a.n_local, [&](int e) { return (a.cnt[e] + kDgChunk - 1) / kDgChunk * nmb; }, P,
                       reinterpret_cast<int32_t*>(smem + L.scan));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = P[a.n_local];
  const int KC = (a.K + kDgBK - 1) / kDgBK;
  const int Ks = a.K / 32;
  const int R2 = 2 * a.R;
  // A K that is not a multiple of 128 ends with a block over [K - 128, K)
  // (e2m1 tensor maps take inner extents in multiples of 128 only; the block
  // stays inside each row), of which the MMA takes the K32 steps past the
  // previous block: k4 >= skip. Its scale bytes: weight word built from
  // groups K/32 - 4 + k4 (id k4); activation word kc holds groups 4kc..
  // (id k4 - skip).
  const int skip = (a.K % kDgBK) ? (kDgBK - a.K % kDgBK) / 32 : 0;
  auto kx = [&](int kc) { return (skip && kc == KC - 1) ? a.K - kDgBK : kc * kDgBK; };
  // Tile t: expert e (the last with P[e] <= t), row block mb, first segment
  // row r0 and live slot count of its chunk.
  auto tile_info = [&](int t, int& e, int& mb, int& r0, int& live) {
    int lo = 0, hi = a.n_local - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (P[mid] <= t) lo = mid; else hi = mid - 1;
    }
    e = lo;
    const int cnt = a.cnt[e];
    const int nch = (cnt + kDgChunk - 1) / kDgChunk;
    const int local = t - P[e];
    mb = local / nch;
    const int c = local % nch;
    r0 = a.seg[e] + kDgChunk * c;
    live = min(kDgChunk, cnt - kDgChunk * c);
  };

  if (warp == 0) {
    if (lane == 0) {
      // -------------------------------------------------------- producer
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
      if (kFp4 && skip) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmWt)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
      int s = 0;
      uint32_t ph = 0;
      int issued[kMaxStages];
      for (int i = 0; i < S; ++i) issued[i] = -1;
      bool ok = true;
      int ti = 0;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++ti) {
        int e, mb, r0, live;
        tile_info(tile, e, mb, r0, live);
        const int n = align16i(live);
        const int m0 = mb * RT;
        if (kFp4) {
          const int tb = ti & 1;
          if (!(ok = wait_phase(tsf_empty(tb), ((ti >> 1) & 1) ^ 1u, abort_flag, a.err))) break;
          const uint32_t dst = sbase + L.tsf + tb * L.tsf_bytes;
          const uint8_t* wexp = a.wsf + (size_t)e * a.rows * Ks;
          if (kGlu && !a.interleaved) {
            const uint32_t vg = (uint32_t)min(128, a.M - m0);
            mbar_arrive_expect_tx(tsf_full(tb), 2u * vg * Ks);
            bulk_load(dst, wexp + (size_t)m0 * Ks, vg * Ks, tsf_full(tb));
            bulk_load(dst + 128u * Ks, wexp + (size_t)(a.M + m0) * Ks, vg * Ks, tsf_full(tb));
          } else {
            const uint32_t rows = kGlu ? 2u * (uint32_t)min(128, a.M - m0) : (uint32_t)min(256, a.M - m0);
            mbar_arrive_expect_tx(tsf_full(tb), rows * Ks);
            bulk_load(dst, wexp + (size_t)(kGlu ? 2 * m0 : m0) * Ks, rows * Ks, tsf_full(tb));
          }
        }
        for (int kc = 0; kc < KC; ++kc) {
          if (!(ok = wait_phase(empty_bar(s), ph ^ 1u, abort_flag, a.err))) break;
          const uint32_t st = sbase + (uint32_t)s * kStBytes;
          mbar_arrive_expect_tx(sfin_bar(s), 2u * n * 4u);
          bulk_load(st + kStSfin, a.asf + (size_t)kc * R2 + 2 * r0, 2u * n * 4u, sfin_bar(s));
          constexpr uint32_t kWBox = kFp4 ? 8192u : 16384u;  // packed global bytes of a 128 x 128 box
          mbar_arrive_expect_tx(full_bar(s), 2u * kWBox + 2u * n * 128u);
          for (int j = 0; j < n / 16; ++j)
            tma_load_2d(st + kStA + 4096u * j, &tmA, kx(kc), 2 * r0 + 32 * j, full_bar(s));
          // e2m1 tail block: its own map based at element K - 128
          const bool tail = kFp4 && skip && kc == KC - 1;
          const CUtensorMap* wm = tail ? &tmWt : &tmW;
          const int xw = tail ? 0 : kx(kc);
          if (kGlu && a.interleaved) {
            tma_load_4d(st + kStB, wm, xw, 0, m0, e, full_bar(s));
            tma_load_4d(st + kStB + 16384u, wm, xw, 1, m0, e, full_bar(s));
          } else if (kGlu) {
            tma_load_4d(st + kStB, wm, xw, m0, 0, e, full_bar(s));
            tma_load_4d(st + kStB + 16384u, wm, xw, m0, 1, e, full_bar(s));
          } else {
            tma_load_4d(st + kStB, wm, xw, m0, 0, e, full_bar(s));
            tma_load_4d(st + kStB + 16384u, wm, xw, m0 + 128, 0, e, full_bar(s));
          }
          issued[s] = (int)ph;
          if (++s == S) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA can exit
        for (int i = 0; i < S; ++i)
          if (issued[i] >= 0) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(full_bar(i), (uint32_t)issued[i]) && globaltimer_ns() - t0 < 2000000ull) {}
          }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------- MMA issuer
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      int ti = 0;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++ti) {
        if (!(ok = wait_phase(acc_empty, (ti & 1) ^ 1u, abort_flag, a.err))) break;
        tc_fence_after();
        for (int kc = 0; kc < KC; ++kc) {
          if (!(ok = wait_phase(full_bar(s), ph, abort_flag, a.err))) break;
          tc_fence_after();
          const uint32_t st = sbase + (uint32_t)s * kStBytes;
          const uint32_t tsf = tmem + 256u + 16u * s;  // A: 4 columns, B: 8 columns
          tc_cp_sf(tsf, desc_sf(st + kStSfa));
          tc_cp_sf(tsf + 4u, desc_sf(st + kStSfb));
          tc_cp_sf(tsf + 8u, desc_sf(st + kStSfb + 512u));
          const int k4_0 = (kc == KC - 1) ? skip : 0;
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            if (k4 < k4_0) continue;
            const uint32_t idesc = dg_idesc(kFp4) | ((uint32_t)k4 << 4) | ((uint32_t)(k4 - k4_0) << 29);
            tc_mma(tmem, desc_sw128(st + kStA + 32u * k4), desc_sw128(st + kStB + 32u * k4), idesc, tsf, tsf + 4u,
                   (kc | (k4 - k4_0)) != 0);
          }
          tc_commit(empty_bar(s));
          if (++s == S) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        tc_commit(acc_full);
      }
      tc_commit(done_bar);
      wait_phase(done_bar, 0, abort_flag, a.err, false);
    }
  } else if (warp == 2) {
    // ------------------------------------------------- scale transposer
    // tcgen05.cp 32x128b.warpx4 takes a 32 x 4 word source in which word
    // (i, j) at 16 i + 4 j holds row 32 j + i; byte b of a word is the scale
    // of the K block's b-th group of 32.
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    int ti = 0;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++ti) {
      int e, mb, r0, live;
      tile_info(tile, e, mb, r0, live);
      const int n2 = 2 * align16i(live);  // activation rows of the tile
      const int m0 = mb * RT;
      const int tb = ti & 1;
      if (kFp4 && !(ok = wait_phase(tsf_full(tb), (ti >> 1) & 1, abort_flag, a.err))) break;
      const uint8_t* tsf = smem + L.tsf + tb * L.tsf_bytes;
      for (int kc = 0; kc < KC; ++kc) {
        if (!(ok = wait_phase(sfin_bar(s), ph, abort_flag, a.err))) break;
        uint8_t* st = stage(s);
        {
          const uint32_t* in = reinterpret_cast<const uint32_t*>(st + kStSfin);
          uint4 v;
          v.x = (lane < n2) ? in[lane] : 0x7F7F7F7Fu;
          v.y = (32 + lane < n2) ? in[32 + lane] : 0x7F7F7F7Fu;
          v.z = (64 + lane < n2) ? in[64 + lane] : 0x7F7F7F7Fu;
          v.w = (96 + lane < n2) ? in[96 + lane] : 0x7F7F7F7Fu;
          *reinterpret_cast<uint4*>(st + kStSfa + 16 * lane) = v;
        }
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          uint32_t w[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            w[j] = 0x7F7F7F7Fu;
            const int r = 32 * j + lane;  // row within the 128-row block
            if (kFp4) {
              // output row of this weight row, and its row in the tile's scale copy
              const int orow = kGlu ? m0 + r : m0 + 128 * blk + r;
              const int raw = kGlu ? (a.interleaved ? 2 * r + blk : 128 * blk + r) : 128 * blk + r;
              if (orow < a.M) {
                const uint8_t* src = tsf + (size_t)raw * Ks + kx(kc) / 32;
                w[j] = (uint32_t)src[0] | ((uint32_t)src[1] << 8) | ((uint32_t)src[2] << 16) |
                       ((uint32_t)src[3] << 24);
              }
            }
          }
          *reinterpret_cast<uint4*>(st + kStSfb + 512 * blk + 16 * lane) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(full_bar(s));
        if (++s == S) { s = 0; ph ^= 1u; }
      }
      if (!ok) break;
      __syncwarp();
      if (kFp4 && lane == 0) mbar_arrive(tsf_empty(tb));
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------- epilogue
    // Warp q holds accumulator lanes 32q..32q+31: lanes j < 16 the hi term
    // and lanes j + 16 the lo term of chunk column 16q + j; shfl_xor 16 sums
    // them.
    const int q = warp & 3;
    int ti = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++ti) {
      int e, mb, r0, live;
      tile_info(tile, e, mb, r0, live);
      const int m0 = mb * RT;
      const float ws = kFp4 ? 1.0f : __ldg(a.wscale + e);
      const uint16_t* bexp = a.bias + (size_t)e * a.rows;
      const int nchunk = min(RT, a.M - m0) / 32;  // 32-row chunks with output rows (M % 32 == 0)
      if (!wait_phase(acc_full, ti & 1, abort_flag, a.err)) break;
      tc_fence_after();
      if (!kGlu) {
        // y2 rows: each low lane finishes its slot's row, 32 outputs per chunk
        const int c = 16 * q + (lane & 15);
        const bool mine = lane < 16 && c < live;
        const int slot = mine ? a.row_slot[r0 + c] : -1;
        const bool any = 16 * q < live;
        for (int ch = 0; any && ch < nchunk; ++ch) {
          uint32_t g[32];
          tmem_ld_32cols(tmem + ((uint32_t)(32 * q) << 16) + 32u * ch, g);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            g[j] = __float_as_uint(__uint_as_float(g[j]) + __shfl_xor_sync(kAll, __uint_as_float(g[j]), 16));
          if (!mine) continue;
          const int r_out = m0 + 32 * ch;
          const uint4* b4 = reinterpret_cast<const uint4*>(bexp + r_out);
          uint4* d = reinterpret_cast<uint4*>(a.y + (size_t)slot * a.rows + r_out);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint4 bv = __ldg(b4 + v);
            const uint32_t* bw = &bv.x;
            uint32_t o[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int j = 8 * v + 2 * t;
              o[t] = pack_bf16x2(fmaf(__uint_as_float(g[j]), ws, bf16_lo(bw[t])),
                                 fmaf(__uint_as_float(g[j + 1]), ws, bf16_hi(bw[t])));
            }
            d[v] = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
        continue;
      }
      // GLU: per pass, the warp holding 16 slots stages their summed gate/up
      // rows in shared memory; then all four warps finish them, lanes over 32
      // consecutive rows (coalesced stores; one warp reduction per group of
      // 32 for the split of act). The accumulator is released after the last
      // pass's reads.
      float* buf = reinterpret_cast<float*>(smem + L.epi);
      const int npass = (live + kEpiSlots - 1) / kEpiSlots;
      for (int p = 0; p < npass; ++p) {
        // slots 8p..8p+7: lanes 8(p % 2) + j (hi) and + 16 (lo) of warp p / 2
        const int lane0 = kEpiSlots * (p & 1);
        if (q == (p >> 1)) {
          for (int ch = 0; ch < nchunk; ++ch) {
            uint32_t g[32], u[32];
            const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16) + 32u * ch;
            tmem_ld_32cols(tq, g);
            tmem_ld_32cols(tq + 128u, u);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float gs = __uint_as_float(g[j]) + __shfl_xor_sync(kAll, __uint_as_float(g[j]), 16);
              const float us = __uint_as_float(u[j]) + __shfl_xor_sync(kAll, __uint_as_float(u[j]), 16);
              if (lane >= lane0 && lane < lane0 + kEpiSlots) {
                buf[(lane - lane0) * kEpiStride + 32 * ch + j] = gs;
                buf[(lane - lane0) * kEpiStride + 128 + 32 * ch + j] = us;
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (p == npass - 1 && lane == 0) mbar_arrive(acc_empty);
        }
        named_barrier(1, 128);
        const int np = min(kEpiSlots, live - kEpiSlots * p);
        for (int sl = q; sl < np; sl += 4) {
          const int col = kEpiSlots * p + sl;  // chunk column
          const int slot = a.row_slot[r0 + col];
          const int srow = r0 + col;
          uint16_t* yrow = a.y + (size_t)slot * a.rows;
          uint32_t wh = 0x7F7F7F7Fu, wl = 0x7F7F7F7Fu;
          for (int ch = 0; ch < nchunk; ++ch) {
            const int i = m0 + 32 * ch + lane;
            const float gsum = buf[sl * kEpiStride + 32 * ch + lane];
            const float usum = buf[sl * kEpiStride + 128 + 32 * ch + lane];
            const int grow = a.interleaved ? 2 * i : i, urow = a.interleaved ? 2 * i + 1 : a.M + i;
            const uint32_t yG = f32_to_bf16_bits(fmaf(gsum, ws, bf16_to_f32(bexp[grow])));
            const uint32_t yU = f32_to_bf16_bits(fmaf(usum, ws, bf16_to_f32(bexp[urow])));
            const uint32_t A = f32_to_bf16_bits(
                glu_value(bf16_to_f32((uint16_t)yG), bf16_to_f32((uint16_t)yU), a.alpha, a.beta, a.limit));
            if (a.interleaved) {
              reinterpret_cast<uint32_t*>(yrow)[i] = yG | (yU << 16);
            } else {
              yrow[grow] = (uint16_t)yG;
              yrow[urow] = (uint16_t)yU;
            }
            a.act[(size_t)slot * a.M + i] = (uint16_t)A;
            // two-term split of the group of 32 act values held by the warp
            const float v = bf16_to_f32((uint16_t)A);
            const float am = __uint_as_float(__reduce_max_sync(kAll, __float_as_uint(fabsf(v))));
            const uint32_t sh = group_scale_byte(am);
            const uint32_t hc = e4m3x2_satfinite(__fmul_rn(v, pow2_f32(127 - (int)sh)), 0.0f) & 0xFFu;
            const float r = __fsub_rn(v, __fmul_rn(e4m3x2_to_f32x2(hc).x, pow2_f32((int)sh - 127)));
            const float ar = __uint_as_float(__reduce_max_sync(kAll, __float_as_uint(fabsf(r))));
            const uint32_t sl2 = group_scale_byte(ar);
            const uint32_t lc = e4m3x2_satfinite(__fmul_rn(r, pow2_f32(127 - (int)sl2)), 0.0f) & 0xFFu;
            a.a_split[(size_t)split_row(srow, 0) * a.M + i] = (uint8_t)hc;
            a.a_split[(size_t)split_row(srow, 1) * a.M + i] = (uint8_t)lc;
            wh = (wh & ~(0xFFu << (8 * ch))) | (sh << (8 * ch));
            wl = (wl & ~(0xFFu << (8 * ch))) | (sl2 << (8 * ch));
          }
          if (lane == 0) {
            a.a_sf[(size_t)mb * R2 + split_row(srow, 0)] = wh;
            a.a_sf[(size_t)mb * R2 + split_row(srow, 1)] = wl;
          }
        }
        named_barrier(1, 128);  // the staging buffer is free for the next pass
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
  }
}

template <bool kFp4, bool kGlu>
cudaError_t set_smem() {
  return cudaFuncSetAttribute(decode_gemm_kernel<kFp4, kGlu>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kSmemMax);
}

// Weight tensor map over [n_local][rows][K] (FP8 bytes, or e2m1 nibbles):
// dims (K, 128-row index, gate/up half, expert). GLU halves: row = half*I + i;
// GLU interleaved: row = 2 i + half (dims 1 and 2 swapped so that the strides
// grow); no GLU: half is a unit dimension. The map covers elements [k0, k0 +
// kext) of each row: e2m1 maps need kext % 128 == 0 and a 32-byte aligned
// start, so MXFP4 takes [0, K - K % 128) and, for a ragged K, a second map
// over [K - 128, K).
bool encode_weights(EncodeTiledFn enc, CUtensorMap* m, const uint8_t* w, bool fp4, int n_local, int rows, int K,
                    int M, bool glu, bool interleaved, int k0, int kext) {
  const uint64_t rb = fp4 ? (uint64_t)K / 2 : (uint64_t)K;
  w += fp4 ? k0 / 2 : k0;
  const uint64_t ex = (uint64_t)rows * rb;
  const CUtensorMapDataType dt = fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  if (glu && interleaved) {
    const uint64_t dims[4] = {(uint64_t)kext, 2, (uint64_t)M, (uint64_t)n_local};
    const uint64_t str[3] = {rb, 2 * rb, ex};
    const uint32_t box[4] = {128, 1, 128, 1};
    return encode_4d(enc, m, dt, w, dims, str, box);
  }
  const uint64_t dims[4] = {(uint64_t)kext, (uint64_t)M, glu ? 2u : 1u, (uint64_t)n_local};
  const uint64_t str[3] = {rb, (uint64_t)M * rb, ex};
  const uint32_t box[4] = {128, 128, 1, 1};
  return encode_4d(enc, m, dt, w, dims, str, box);
}

}  // namespace

DecodeWs decode_ws_layout(int T, int k, int H, int I, int n_local) {
  DecodeWs w{};
  const long S = (long)T * k;
  const long R = ((S + 15L * lmin(n_local, S)) + 15) / 16 * 16;
  w.R = (int)lmax(R, 16);
  const long KCx = (H + 127) / 128, KCa = (I + 127) / 128;
  auto up = [](size_t v) { return (v + 1023) / 1024 * 1024; };
  size_t off = 0;
  w.cnt = off;      off = up(off + (size_t)n_local * 4);
  w.seg = off;      off = up(off + (size_t)n_local * 4);
  w.row_slot = off; off = up(off + (size_t)w.R * 4);
  w.xs = off;       off = up(off + 2 * (size_t)w.R * H);
  w.xsf = off;      off = up(off + 2 * (size_t)KCx * w.R * 4);
  w.as = off;       off = up(off + 2 * (size_t)w.R * I);
  w.asf = off;      off = up(off + 2 * (size_t)KCa * w.R * 4);
  w.total = off;
  return w;
}

bool decode_gemm_ok(int T, int k, int H, int I, int n_local, int wfmt) {
  const long S = (long)T * k;
  if (T < 1 || T > 128 || S > kDgMaxSlots || n_local < 1 || n_local > kDgMaxLocal) return false;
  if (H % 32 != 0 || I % 32 != 0 || H < kDgBK || I < kDgBK) return false;
  // MXFP4: the ragged-K map starts at byte (K - 128) / 2, 32-byte aligned
  if (wfmt == MOE_WFMT_MXFP4_G32 && (H / 32 > kDgMaxKs || I / 32 > kDgMaxKs || H % 64 || I % 64)) return false;
  const bool fp4 = wfmt == MOE_WFMT_MXFP4_G32;
  if (dg_layout(fp4, H / 32).stages < 2 || dg_layout(fp4, I / 32).stages < 2) return false;
  return true;
}

cudaError_t init_decode_gemm() {
  cudaError_t ce;
  if ((ce = set_smem<false, true>()) != cudaSuccess) return ce;
  if ((ce = set_smem<false, false>()) != cudaSuccess) return ce;
  if ((ce = set_smem<true, true>()) != cudaSuccess) return ce;
  return set_smem<true, false>();
}

int launch_decode_gemm(const moe_decode_args& a, EncodeTiledFn enc, int num_sms, uint32_t* err, cudaStream_t st) {
  const bool fp4 = a.wfmt == MOE_WFMT_MXFP4_G32;
  const DecodeWs L = decode_ws_layout(a.T, a.k, a.H, a.I, a.num_local_experts);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  int32_t* cnt = reinterpret_cast<int32_t*>(ws + L.cnt);
  int32_t* seg = reinterpret_cast<int32_t*>(ws + L.seg);
  int32_t* row_slot = reinterpret_cast<int32_t*>(ws + L.row_slot);
  uint8_t* xs = ws + L.xs;
  uint32_t* xsf = reinterpret_cast<uint32_t*>(ws + L.xsf);
  uint8_t* as = ws + L.as;
  uint32_t* asf = reinterpret_cast<uint32_t*>(ws + L.asf);
  const int n_local = a.num_local_experts;

  CUtensorMap mW1, mW1t, mB1, mW2, mW2t, mB2;
  const bool il = a.glu_layout == MOE_GLU_INTERLEAVED;
  const int H = a.H, I = a.I;
  const int ext1 = fp4 ? H - H % kDgBK : H, ext2 = fp4 ? I - I % kDgBK : I;
  if (!encode_weights(enc, &mW1, a.w_gu, fp4, n_local, 2 * I, H, I, true, il, 0, ext1) ||
      !encode_weights(enc, &mW2, a.w_d, fp4, n_local, H, I, H, false, false, 0, ext2) ||
      !encode_weights(enc, &mW1t, a.w_gu, fp4, n_local, 2 * I, H, I, true, il, fp4 && H % kDgBK ? H - kDgBK : 0,
                      fp4 && H % kDgBK ? kDgBK : ext1) ||
      !encode_weights(enc, &mW2t, a.w_d, fp4, n_local, H, I, H, false, false, fp4 && I % kDgBK ? I - kDgBK : 0,
                      fp4 && I % kDgBK ? kDgBK : ext2) ||
      !encode_2d(enc, &mB1, CU_TENSOR_MAP_DATA_TYPE_UINT8, xs, (uint64_t)a.H, 2 * (uint64_t)L.R, (uint64_t)a.H,
                 kDgBK, 32) ||
      !encode_2d(enc, &mB2, CU_TENSOR_MAP_DATA_TYPE_UINT8, as, (uint64_t)a.I, 2 * (uint64_t)L.R, (uint64_t)a.I,
                 kDgBK, 32))
    return MOE_ERR_INVALID_ARG;

  DsArgs ds{};
  ds.ids = a.topk_ids;
  ds.T = a.T;
  ds.k = a.k;
  ds.expert_start = a.expert_start;
  ds.n_local = n_local;
  ds.x = a.x;
  ds.H = a.H;
  ds.cnt = cnt;
  ds.seg = seg;
  ds.row_slot = row_slot;
  ds.xs = xs;
  ds.xsf = xsf;
  ds.R = L.R;
  const int S = a.T * a.k;
  const long items = (long)S * ((a.H + kDgBK - 1) / kDgBK);  // one warp each
  const int gsplit = (int)lmax(1, lmin((items + 7) / 8, 8L * num_sms));
  decode_split_kernel<<<gsplit, 256, 0, st>>>(ds);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;

  DgArgs g{};
  g.cnt = cnt;
  g.seg = seg;
  g.row_slot = row_slot;
  g.n_local = n_local;
  g.R = L.R;
  g.err = err;
  g.alpha = a.glu_alpha;
  g.beta = a.glu_beta;
  g.limit = a.glu_limit;
  // GEMM 1 + GLU + split of act
  g.asf = xsf;
  g.wsf = a.w_gu_sf;
  g.wscale = a.w_gu_scale;
  g.bias = a.b_gu;
  g.K = a.H;
  g.M = a.I;
  g.rows = 2 * a.I;
  g.interleaved = il;
  g.y = a.y1;
  g.act = a.act;
  g.a_split = as;
  g.a_sf = asf;
  g.lay = dg_layout(fp4, a.H / 32);
  cudaError_t ce = fp4 ? launch_maybe_pdl(decode_gemm_kernel<true, true>, dim3(num_sms), dim3(kDgThreads),
                                          (size_t)g.lay.bytes, st, true, mW1, mW1t, mB1, g)
                       : launch_maybe_pdl(decode_gemm_kernel<false, true>, dim3(num_sms), dim3(kDgThreads),
                                          (size_t)g.lay.bytes, st, true, mW1, mW1t, mB1, g);
  if (ce != cudaSuccess) return MOE_ERR_CUDA;
  // GEMM 2
  g.asf = asf;
  g.wsf = a.w_d_sf;
  g.wscale = a.w_d_scale;
  g.bias = a.b_d;
  g.K = a.I;
  g.M = a.H;
  g.rows = a.H;
  g.interleaved = 0;
  g.y = a.y2;
  g.act = nullptr;
  g.a_split = nullptr;
  g.a_sf = nullptr;
  g.lay = dg_layout(fp4, a.I / 32);
  ce = fp4 ? launch_maybe_pdl(decode_gemm_kernel<true, false>, dim3(num_sms), dim3(kDgThreads), (size_t)g.lay.bytes,
                              st, true, mW2, mW2t, mB2, g)
           : launch_maybe_pdl(decode_gemm_kernel<false, false>, dim3(num_sms), dim3(kDgThreads), (size_t)g.lay.bytes,
                              st, true, mW2, mW2t, mB2, g);
  if (ce != cudaSuccess) return MOE_ERR_CUDA;
  return launch_weighted_sum(a, true, st) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
