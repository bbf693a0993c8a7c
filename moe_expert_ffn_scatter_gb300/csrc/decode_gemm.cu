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
// Operands of tcgen05.mma.kind::mxf8f6f4.block_scale (M128, N = the expert's
// slots rounded up to 16, at most 64 per tile, K32): the weights are the A
// operand, 128 rows per tile, moved by TMA in their stored format (e4m3, or
// e2m1 expanded to a byte per element by the 16U4_ALIGN16B tensor-map type)
// with their UE8M0 group-32 scales -- FP8-per-expert weights take unit scales
// and their fp32 scale in the epilogue; the slots are the B operand.
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
//             tile), then per 128-wide K block the B terms' scale words (bulk)
//             and the A (gate and up blocks with GLU) and B tiles (TMA)
//   warp 1    TMEM owner and MMA issuer (two accumulators of 64 columns per
//             buffer, double-buffered)
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
constexpr int kDgChunk = 64;  // slot columns per tile
constexpr int kDgAlign = 16;  // segment starts and the MMA's N granularity
constexpr int kDgMaxLocal = 1024;
constexpr int kDgMaxSlots = 4096;
constexpr int kDgMaxKs = 128;  // MXFP4 scale bytes per weight row (K <= 4096)
constexpr int kDgBK = 128;

// Stage layout (bytes): two 128 x 128 A blocks (gate, up), two 64 x 128 B
// terms (hi, lo), the tcgen05.cp sources of the A and B scales, and the B
// scale words as copied (row-major, 64 per term).
constexpr uint32_t kStA0 = 0, kStA1 = 16384, kStB0 = 32768, kStB1 = 40960;
constexpr uint32_t kStSfa = 49152;   // + 512 * block
constexpr uint32_t kStSfb = 50176;   // + 512 * term
constexpr uint32_t kStSfin = 51200;  // + 256 * term
constexpr uint32_t kStBytes = 52224;  // 51 KB, keeps every stage 1024-byte aligned

template <bool kFp4>
struct DgSmem {
  static constexpr int kStages = kFp4 ? 3 : 4;
  static constexpr uint32_t kTsf = kStages * kStBytes;                        // 2 x 256 rows x Ks (MXFP4)
  static constexpr uint32_t kTsfBytes = kFp4 ? 256u * kDgMaxKs : 0u;
  static constexpr uint32_t kPrefix = kTsf + 2 * kTsfBytes;                   // tile prefix [n_local + 1]
  static constexpr uint32_t kBar = kPrefix + (kDgMaxLocal + 1) * 4 + 4;       // 8-byte aligned
  static constexpr uint32_t kNumBars = 3 * kStages + 9;
  static constexpr uint32_t kTmemSlot = kBar + kNumBars * 8;
  static constexpr uint32_t kAbort = kTmemSlot + 4;
  static constexpr uint32_t kScan = kAbort + 4;                               // [32] scan scratch
  static constexpr uint32_t kUsed = kScan + 32 * 4;
  static constexpr uint32_t kBytes = kUsed + 1024;
  static_assert(kBytes <= 232448, "shared memory budget");
  static_assert(kBar % 8 == 0, "mbarrier alignment");
};

__host__ __device__ constexpr int align16i(int v) { return (v + kDgAlign - 1) / kDgAlign * kDgAlign; }

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

// Two-term split of one group of 32 values, one per lane (warp-collective):
// codes of the hi and lo terms of this lane's value and the group's two scale
// bytes.
__device__ __forceinline__ void split_group(float v, uint32_t& ch, uint32_t& cl, uint32_t& sh, uint32_t& sl) {
  const float a = __uint_as_float(__reduce_max_sync(kAll, __float_as_uint(fabsf(v))));
  sh = group_scale_byte(a);
  ch = e4m3x2_satfinite(__fmul_rn(v, pow2_f32(127 - (int)sh)), 0.0f) & 0xFFu;
  const float r = __fsub_rn(v, __fmul_rn(e4m3x2_to_f32x2(ch).x, pow2_f32((int)sh - 127)));
  const float ar = __uint_as_float(__reduce_max_sync(kAll, __float_as_uint(fabsf(r))));
  sl = group_scale_byte(ar);
  cl = e4m3x2_satfinite(__fmul_rn(r, pow2_f32(127 - (int)sl)), 0.0f) & 0xFFu;
}

struct DsArgs {
  const int32_t* ids;
  int T, k, expert_start, n_local;
  const uint16_t* x;  // [T][H]
  int H;
  int32_t* cnt;       // [n_local]
  int32_t* seg;       // [n_local]
  int32_t* row_slot;  // [R]
  uint8_t* xs;        // [2][R][H]
  uint32_t* xsf;      // [2][ceil(H/128)][R]
  int R;
};

// Segments and the split of x. Every CTA derives the same counts, segment
// starts and per-slot ranks from topk_ids (the rank of a slot is the number
// of earlier slots with the same expert, so the order is deterministic); CTA
// 0 writes the counts, the starts and the padding entries of row_slot; each
// warp then takes whole slots: their row_slot entry and the split x row.
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
  const int H = a.H, G = H / 32, W = (H + kDgBK - 1) / kDgBK;
  for (int s = blockIdx.x * 8 + warp; s < S; s += gridDim.x * 8) {
    const int lid = lid_s[s];
    if (lid < 0) continue;  // warp-uniform
    int c = 0;
    for (int s2 = lane; s2 < s; s2 += 32) c += (lid_s[s2] == lid);
    c = __reduce_add_sync(kAll, c);
    const int row = seg_s[lid] + c;
    if (lane == 0) a.row_slot[row] = s;
    const uint16_t* src = a.x + (size_t)(s / a.k) * H;
    uint8_t* hrow = a.xs + (size_t)row * H;
    uint8_t* lrow = a.xs + ((size_t)a.R + row) * H;
    for (int w = 0; w < W; ++w) {
      uint32_t wh = 0x7F7F7F7Fu, wl = 0x7F7F7F7Fu;  // groups past H keep unit scales
      for (int b = 0; b < 4; ++b) {
        const int g = 4 * w + b;
        if (g >= G) break;
        uint32_t ch, cl, sh, sl;
        split_group(bf16_to_f32(src[32 * g + lane]), ch, cl, sh, sl);
        hrow[32 * g + lane] = (uint8_t)ch;
        lrow[32 * g + lane] = (uint8_t)cl;
        wh = (wh & ~(0xFFu << (8 * b))) | (sh << (8 * b));
        wl = (wl & ~(0xFFu << (8 * b))) | (sl << (8 * b));
      }
      if (lane == 0) {
        a.xsf[(size_t)w * a.R + row] = wh;
        a.xsf[((size_t)W + w) * a.R + row] = wl;
      }
    }
  }
}

struct DgArgs {
  const int32_t* cnt;       // [n_local] slots per local expert
  const int32_t* seg;       // [n_local] first segment row of the expert
  const int32_t* row_slot;  // [R] slot t*k+j of each segment row, -1 for padding
  int n_local, R;
  const uint32_t* bsf;  // [2][KC][R] scale words of the B terms
  const uint8_t* wsf;   // MXFP4: [n_local][rows][K/32]
  const float* wscale;  // FP8: [n_local]
  const uint16_t* bias;  // [n_local][rows]
  int K, M, rows;        // reduction length; output rows (I with GLU, else H); weight rows per expert
  int interleaved;
  float alpha, beta, limit;
  uint16_t* y;        // [T*k][rows]
  uint16_t* act;      // GLU: [T*k][M]
  uint8_t* a_split;   // GLU: [2][R][M] e4m3 terms of act
  uint32_t* a_sf;     // GLU: [2][ceil(M/128)][R]
  uint32_t* err;
};

// Instruction descriptor: A format e2m1 (5) or e4m3 (0), B e4m3, K-major, N
// >> 3 at bit 17, UE8M0 scales (bit 23), M = 128 (M >> 4 at bit 24); the
// scale-factor ids (B at bit 4, A at bit 29) are or-ed in per K32 step.
__device__ __forceinline__ uint32_t dg_idesc(bool a_fp4, int n) {
  return ((a_fp4 ? 5u : 0u) << 7) | ((uint32_t)(n >> 3) << 17) | (1u << 23) | ((uint32_t)(128 >> 4) << 24);
}

template <bool kFp4, bool kGlu>
__global__ void __launch_bounds__(kDgThreads, 1) decode_gemm_kernel(const __grid_constant__ CUtensorMap tmW,
                                                                    const __grid_constant__ CUtensorMap tmWt,
                                                                    const __grid_constant__ CUtensorMap tmB,
                                                                    const __grid_constant__ DgArgs a) {
  using L = DgSmem<kFp4>;
  constexpr int S = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  int32_t* P = reinterpret_cast<int32_t*>(smem + L::kPrefix);
  const uint32_t bar0 = sbase + L::kBar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto sfin_bar = [&](int s) { return bar0 + 8u * (2 * S + s); };
  auto tsf_full = [&](int b) { return bar0 + 8u * (3 * S + b); };
  auto tsf_empty = [&](int b) { return bar0 + 8u * (3 * S + 2 + b); };
  auto acc_full = [&](int b) { return bar0 + 8u * (3 * S + 4 + b); };
  auto acc_empty = [&](int b) { return bar0 + 8u * (3 * S + 6 + b); };
  const uint32_t done_bar = bar0 + 8u * (3 * S + 8);
  auto stage = [&](int s) { return smem + (size_t)s * kStBytes; };

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 2);   // producer's expect_tx arrive + transposer's arrive
      mbar_init(empty_bar(s), 1);  // tcgen05.commit
      mbar_init(sfin_bar(s), 1);   // producer's expect_tx arrive for the B scale words
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tsf_full(b), 1);
      mbar_init(tsf_empty(b), 1);
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), 4);  // one arrive per epilogue warp
    }
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
  // The segments, the B terms and (second GEMM) the act terms come from the
  // preceding kernels of the stream.
  pdl_wait();
  const int nmb = (a.M + 127) / 128;
  block_exclusive_scan(a.n_local, [&](int e) { return (a.cnt[e] + kDgChunk - 1) / kDgChunk * nmb; }, P,
                       reinterpret_cast<int32_t*>(smem + L::kScan));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = P[a.n_local];
  const int KC = (a.K + kDgBK - 1) / kDgBK;
  const int Ks = a.K / 32;
  // A K that is not a multiple of 128 ends with a block over [K - 128, K)
  // (e2m1 tensor maps take inner extents in multiples of 128 only; the block
  // stays inside each row), of which the MMA takes the K32 steps past the
  // previous block: k4 >= skip. Its scale bytes: A word built from groups
  // K/32 - 4 + k4 (id k4); B word kc holds groups 4kc.. (id k4 - skip).
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
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
      int s = 0;
      uint32_t ph = 0;
      int issued[S];
      for (int i = 0; i < S; ++i) issued[i] = -1;
      bool ok = true;
      int ti = 0;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++ti) {
        int e, mb, r0, live;
        tile_info(tile, e, mb, r0, live);
        const int n = align16i(live);
        const int m0 = mb * 128;
        if (kFp4) {
          const int tb = ti & 1;
          if (!(ok = wait_phase(tsf_empty(tb), ((ti >> 1) & 1) ^ 1u, abort_flag, a.err))) break;
          const uint32_t dst = sbase + L::kTsf + tb * L::kTsfBytes;
          const uint32_t vg = (uint32_t)min(128, a.M - m0);
          const uint8_t* wexp = a.wsf + (size_t)e * a.rows * Ks;
          if (kGlu && !a.interleaved) {
            mbar_arrive_expect_tx(tsf_full(tb), 2u * vg * Ks);
            bulk_load(dst, wexp + (size_t)m0 * Ks, vg * Ks, tsf_full(tb));
            bulk_load(dst + 128u * Ks, wexp + (size_t)(a.M + m0) * Ks, vg * Ks, tsf_full(tb));
          } else {
            const uint32_t rows = kGlu ? 2u * vg : vg;
            mbar_arrive_expect_tx(tsf_full(tb), rows * Ks);
            bulk_load(dst, wexp + (size_t)(kGlu ? 2 * m0 : m0) * Ks, rows * Ks, tsf_full(tb));
          }
        }
        for (int kc = 0; kc < KC; ++kc) {
          if (!(ok = wait_phase(empty_bar(s), ph ^ 1u, abort_flag, a.err))) break;
          const uint32_t st = sbase + (uint32_t)s * kStBytes;
          mbar_arrive_expect_tx(sfin_bar(s), 2u * n * 4u);
          bulk_load(st + kStSfin, a.bsf + (size_t)kc * a.R + r0, n * 4u, sfin_bar(s));
          bulk_load(st + kStSfin + 256u, a.bsf + ((size_t)KC + kc) * a.R + r0, n * 4u, sfin_bar(s));
          constexpr uint32_t kWBox = kFp4 ? 8192u : 16384u;  // packed global bytes of a 128 x 128 box
          mbar_arrive_expect_tx(full_bar(s), (kGlu ? 2u : 1u) * kWBox + 2u * n * 128u);
          // e2m1 tail block: its own map based at element K - 128
          const bool tail = kFp4 && skip && kc == KC - 1;
          const CUtensorMap* wm = tail ? &tmWt : &tmW;
          const int xa = tail ? 0 : kx(kc);
          if (kGlu && a.interleaved) {
            tma_load_4d(st + kStA0, wm, xa, 0, m0, e, full_bar(s));
            tma_load_4d(st + kStA1, wm, xa, 1, m0, e, full_bar(s));
          } else {
            tma_load_4d(st + kStA0, wm, xa, m0, 0, e, full_bar(s));
            if (kGlu) tma_load_4d(st + kStA1, wm, xa, m0, 1, e, full_bar(s));
          }
          for (int j = 0; j < n / 16; ++j) {
            tma_load_2d(st + kStB0 + 2048u * j, &tmB, kx(kc), r0 + 16 * j, full_bar(s));
            tma_load_2d(st + kStB1 + 2048u * j, &tmB, kx(kc), a.R + r0 + 16 * j, full_bar(s));
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
        int e, mb, r0, live;
        tile_info(tile, e, mb, r0, live);
        const int n = align16i(live);
        const int b = ti & 1;
        if (!(ok = wait_phase(acc_empty(b), ((ti >> 1) & 1) ^ 1u, abort_flag, a.err))) break;
        tc_fence_after();
        const uint32_t dg = tmem + 128u * b, du = dg + 64u;
        const uint32_t ibase = dg_idesc(kFp4, n);
        for (int kc = 0; kc < KC; ++kc) {
          if (!(ok = wait_phase(full_bar(s), ph, abort_flag, a.err))) break;
          tc_fence_after();
          const uint32_t st = sbase + (uint32_t)s * kStBytes;
          const uint32_t tsf = tmem + 256u + 32u * s;  // A gate, A up, B hi, B lo: 4 columns each
          tc_cp_sf(tsf, desc_sf(st + kStSfa));
          if (kGlu) tc_cp_sf(tsf + 4u, desc_sf(st + kStSfa + 512u));
          tc_cp_sf(tsf + 8u, desc_sf(st + kStSfb));
          tc_cp_sf(tsf + 12u, desc_sf(st + kStSfb + 512u));
          const int k4_0 = (kc == KC - 1) ? skip : 0;
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            if (k4 < k4_0) continue;
            const uint32_t idesc = ibase | ((uint32_t)(k4 - k4_0) << 4) | ((uint32_t)k4 << 29);
#pragma unroll
            for (int p = 0; p < 2; ++p) {
              const uint64_t db = desc_sw128(st + (p ? kStB1 : kStB0) + 32u * k4);
              const uint32_t acc = (kc | (k4 - k4_0) | p) != 0;
              tc_mma(dg, desc_sw128(st + kStA0 + 32u * k4), db, idesc, tsf, tsf + 8u + 4u * p, acc);
              if (kGlu) tc_mma(du, desc_sw128(st + kStA1 + 32u * k4), db, idesc, tsf + 4u, tsf + 8u + 4u * p, acc);
            }
          }
          tc_commit(empty_bar(s));
          if (++s == S) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        tc_commit(acc_full(b));
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
      const int n = align16i(live);
      const int m0 = mb * 128;
      const int tb = ti & 1;
      if (kFp4 && !(ok = wait_phase(tsf_full(tb), (ti >> 1) & 1, abort_flag, a.err))) break;
      const uint8_t* tsf = smem + L::kTsf + tb * L::kTsfBytes;
      for (int kc = 0; kc < KC; ++kc) {
        if (!(ok = wait_phase(sfin_bar(s), ph, abort_flag, a.err))) break;
        uint8_t* st = stage(s);
#pragma unroll
        for (int p = 0; p < 2; ++p) {
          const uint32_t* in = reinterpret_cast<const uint32_t*>(st + kStSfin + 256 * p);
          uint4 v;
          v.x = (lane < n) ? in[lane] : 0x7F7F7F7Fu;
          v.y = (32 + lane < n) ? in[32 + lane] : 0x7F7F7F7Fu;
          v.z = 0x7F7F7F7Fu;
          v.w = 0x7F7F7F7Fu;
          *reinterpret_cast<uint4*>(st + kStSfb + 512 * p + 16 * lane) = v;
        }
#pragma unroll
        for (int blk = 0; blk < (kGlu ? 2 : 1); ++blk) {
          uint32_t w[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            w[j] = 0x7F7F7F7Fu;
            const int r = 32 * j + lane;
            if (kFp4 && m0 + r < a.M) {
              const int raw = kGlu ? (a.interleaved ? 2 * r + blk : 128 * blk + r) : r;
              const uint8_t* src = tsf + (size_t)raw * Ks;
              uint32_t word = 0;
              const int g0 = kx(kc) / 32;
#pragma unroll
              for (int bb = 0; bb < 4; ++bb) word |= (uint32_t)src[g0 + bb] << (8 * bb);
              w[j] = word;
            }
          }
          *reinterpret_cast<uint4*>(st + kStSfa + 512 * blk + 16 * lane) = make_uint4(w[0], w[1], w[2], w[3]);
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
    const int q = warp & 3;
    const int KC2 = (a.M + kDgBK - 1) / kDgBK;  // scale words per act row (GLU)
    int ti = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++ti) {
      int e, mb, r0, live;
      tile_info(tile, e, mb, r0, live);
      const int b = ti & 1;
      const int i = mb * 128 + 32 * q + lane;  // output row of this thread
      const bool valid = i < a.M;
      const int slot_lo = a.row_slot[r0 + lane];
      const int slot_hi = (live > 32) ? a.row_slot[r0 + 32 + lane] : -1;
      const float ws = kFp4 ? 1.0f : __ldg(a.wscale + e);
      const uint16_t* bexp = a.bias + (size_t)e * a.rows;
      const int grow = kGlu ? (a.interleaved ? 2 * i : i) : i;
      const int urow = a.interleaved ? 2 * i + 1 : a.M + i;
      const float bg = valid ? bf16_to_f32(bexp[grow]) : 0.0f;
      const float bu = (kGlu && valid) ? bf16_to_f32(bexp[urow]) : 0.0f;
      if (!wait_phase(acc_full(b), (ti >> 1) & 1, abort_flag, a.err)) break;
      tc_fence_after();
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        if (32 * h >= live) break;
        uint32_t g[32], u[32];
        const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + 128u * b + 32u * h;
        tmem_ld_32cols(tbase, g);
        if (kGlu) tmem_ld_32cols(tbase + 64u, u);
        tmem_ld_wait();
        if (h == 1 || live <= 32) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_empty(b));
        }
        const int slot_src = h ? slot_hi : slot_lo;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (32 * h + c >= live) break;  // warp-uniform
          const int slot = __shfl_sync(kAll, slot_src, c);
          const size_t yrow = (size_t)slot * a.rows;
          if (kGlu) {
            const uint32_t yg = f32_to_bf16_bits(fmaf(__uint_as_float(g[c]), ws, bg));
            const uint32_t yu = f32_to_bf16_bits(fmaf(__uint_as_float(u[c]), ws, bu));
            const uint32_t av =
                f32_to_bf16_bits(glu_value(bf16_to_f32((uint16_t)yg), bf16_to_f32((uint16_t)yu), a.alpha, a.beta,
                                           a.limit));
            if (valid) {
              if (a.interleaved) {
                *reinterpret_cast<uint32_t*>(a.y + yrow + grow) = yg | (yu << 16);
              } else {
                a.y[yrow + grow] = (uint16_t)yg;
                a.y[yrow + urow] = (uint16_t)yu;
              }
              a.act[(size_t)slot * a.M + i] = (uint16_t)av;
            }
            uint32_t ch, cl, sh, sl;
            split_group(valid ? bf16_to_f32((uint16_t)av) : 0.0f, ch, cl, sh, sl);
            const int row = r0 + 32 * h + c;
            if (valid) {
              a.a_split[(size_t)row * a.M + i] = (uint8_t)ch;
              a.a_split[((size_t)a.R + row) * a.M + i] = (uint8_t)cl;
            }
            if (lane == 0) {
              reinterpret_cast<uint8_t*>(a.a_sf + (size_t)mb * a.R + row)[q] = (uint8_t)sh;
              reinterpret_cast<uint8_t*>(a.a_sf + ((size_t)KC2 + mb) * a.R + row)[q] = (uint8_t)sl;
            }
          } else if (valid) {
            a.y[yrow + i] = (uint16_t)f32_to_bf16_bits(fmaf(__uint_as_float(g[c]), ws, bg));
          }
        }
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
                              (int)DgSmem<kFp4>::kBytes);
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
                 kDgBK, 16) ||
      !encode_2d(enc, &mB2, CU_TENSOR_MAP_DATA_TYPE_UINT8, as, (uint64_t)a.I, 2 * (uint64_t)L.R, (uint64_t)a.I,
                 kDgBK, 16))
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
  const int gsplit = (int)lmax(1, lmin((S + 7) / 8, num_sms));
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
  g.bsf = xsf;
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
  cudaError_t ce = fp4 ? launch_maybe_pdl(decode_gemm_kernel<true, true>, dim3(num_sms), dim3(kDgThreads),
                                          DgSmem<true>::kBytes, st, true, mW1, mW1t, mB1, g)
                       : launch_maybe_pdl(decode_gemm_kernel<false, true>, dim3(num_sms), dim3(kDgThreads),
                                          DgSmem<false>::kBytes, st, true, mW1, mW1t, mB1, g);
  if (ce != cudaSuccess) return MOE_ERR_CUDA;
  // GEMM 2
  g.bsf = asf;
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
  ce = fp4 ? launch_maybe_pdl(decode_gemm_kernel<true, false>, dim3(num_sms), dim3(kDgThreads), DgSmem<true>::kBytes,
                              st, true, mW2, mW2t, mB2, g)
           : launch_maybe_pdl(decode_gemm_kernel<false, false>, dim3(num_sms), dim3(kDgThreads),
                              DgSmem<false>::kBytes, st, true, mW2, mW2t, mB2, g);
  if (ce != cudaSuccess) return MOE_ERR_CUDA;
  return launch_weighted_sum(a, true, st) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
