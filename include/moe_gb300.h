/*
 * moe_gb300.h -- C ABI of the GB300 (sm_103a) routed MoE expert FFN library.
 *
 * The hot path: top-k routing -> token scatter that writes aligned prefix-sum
 * expert endpoints -> grouped GEMM1 (w13, gate/up) -> SiLU*mul with e4m3
 * quantisation and packed UE8M0 scales over live rows only -> grouped GEMM2
 * (w2, down) -> top-k weighted combine; plus the small-batch sparse GEMV
 * decode variant.
 *
 * Sources, cited by tag and the page's own section:
 *  [LR] "Blackwell FP4 MoE：把 live-row 边界贯穿整个 FFN"
 *  [DG] "Blackwell 上的 DeepGEMM FusedMoE（sglang）"
 *  [SD] "Phase 20: Sparse MoE Decode — 只算被路由到的专家"
 *  [KM] "kimi3_pro6000_sglang_sm120_flashinfer_mxfp4" experiment log
 *
 * Conventions (all entry points)
 *  - Plain C: pointers and sizes only. Pointers named in argument structs are
 *    DEVICE pointers unless marked "host". Row-major unless stated.
 *  - Ownership: the caller allocates and owns every buffer, including the
 *    capacity workspaces; the library never allocates on the hot path, keeps
 *    no pointer after a call returns and never returns aliases. (Only
 *    moe_ctx_create allocates: the context, its 4-byte device error word and
 *    a 256 KB table of SiLU over all bf16 values, filled once on the device.)
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and enqueue a fixed launch structure that depends on the
 *    sizes only, never on routing counts: every call may be captured into a
 *    CUDA graph and replayed while the device contents change ([LR] §3).
 *  - Status: 0 on success; a negative MOE_ERR_* code otherwise. Arguments are
 *    validated on the host before anything is enqueued; an invalid argument
 *    enqueues nothing. Anomalies that only the device can see (an expert id
 *    out of range, a capacity overflow, a pipeline wait that ran out) set bits
 *    in the context's device error word (moe_get_device_error); nothing traps.
 *  - Number formats: bf16 as uint16 bit patterns; e4m3 codes as uint8 (OCP
 *    FP8 E4M3, largest finite 448); e2m1 packed two per byte with the LOW
 *    nibble holding the even index; UE8M0 scale bytes b meaning 2^(b-127).
 *  - "Packed activation scales" (ASF): int32 array [ceil(G/4)][ld] with
 *    ld = align4(rows) ("MN-major"): byte (g % 4) of word [g/4][row] is the
 *    scale of the row's 128-column group g; unused bytes of the last word of a
 *    written row are 0 ([DG] §2.4.1 and 附录 A: 4 uint8 per int32 along K,
 *    MN-major).
 *  - Endpoints: expert_ends[e] is the real (unaligned) end of expert e's rows;
 *    start[0] = 0, start[e] = align_up(expert_ends[e-1], A) ([LR] §2). Rows
 *    outside [start[e], expert_ends[e]) are padding: no kernel writes them.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef struct moe_ctx moe_ctx;
typedef void* moe_stream_t; /* cudaStream_t */

/* status codes */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)
#define MOE_ERR_CAPACITY (-2)
#define MOE_ERR_UNSUPPORTED (-3)
#define MOE_ERR_CUDA (-4)
#define MOE_ERR_DEVICE (-5)

/* device error bits */
#define MOE_DEVERR_EXPERT_ID 0x1u      /* an expert id outside [0, E) reached a kernel that needs it */
#define MOE_DEVERR_CAPACITY 0x2u       /* expert_ends[E-1] > cap seen on the device */
#define MOE_DEVERR_WAIT_TIMEOUT 0x4u   /* a bounded pipeline wait in a GEMM ran out */
#define MOE_DEVERR_ENDPOINTS 0x8u      /* expert_ends not non-decreasing / beyond capacity */

/* routing modes */
#define MOE_ROUTE_SOFTMAX_TOPK 0       /* softmax -> top-k -> renormalise */
#define MOE_ROUTE_SIGMOID_BIAS_TOPK 1  /* select on sigmoid + bias, weights from unbiased sigmoid */
#define MOE_ROUTE_PRECOMPUTED 2        /* topk_ids given by the caller */

/* activation kinds between the GEMMs */
#define MOE_ACT_SILU 0                 /* h = silu(gate) * up */
#define MOE_ACT_SILU_CLAMP 1           /* gate = min(gate, L); up = clamp(up, -L, L) first */
#define MOE_ACT_SITU 2                 /* h = (bs tanh(g/bs) sigmoid(g)) * (bl tanh(u/bl)) */

/* decode weight formats */
#define MOE_WFMT_FP8_PER_EXPERT 0      /* e4m3 [E,N,K] + fp32 scale [E] */
#define MOE_WFMT_MXFP4_G32 1           /* e2m1 [E,N,K/2] + UE8M0 [E,N,K/32] */

/* decode GLU layouts of the gate_up output */
#define MOE_GLU_HALVES 0               /* [gate_0..gate_{I-1}, up_0..up_{I-1}] */
#define MOE_GLU_INTERLEAVED 1          /* [gate_0, up_0, gate_1, up_1, ...] */

/* decode paths (moe_decode_args.path) */
#define MOE_DECODE_AUTO 0              /* by size and workspace, see moe_sparse_gemv_decode */
#define MOE_DECODE_TCGEN05 1           /* block-scaled tcgen05 path (workspace required) */
#define MOE_DECODE_MMA_SYNC 2          /* m16n8k16 path (T <= 8) */
#define MOE_DECODE_GEMV 3              /* one GEMV block per (token, slot, 32 rows) */

/* ------------------------------------------------------------- context
 * moe_ctx_create: binds `device`, reads its SM count, allocates the 4-byte
 *   device error word and the SiLU table (entry i = silu of the bf16 value
 *   with bits i under the library's exp specification; the activation step
 *   looks SiLU up there, its input being a bf16 gate value). It also sets up
 *   the grouped GEMM: the number of CTA pairs of its two-SM kernel that the
 *   device runs at once (cluster occupancy). A grouped GEMM call takes the
 *   two-SM kernel when E <= 1024 and the capacity holds at least 160 routed
 *   rows per expert (cap - 127 E >= 160 E), else the one-CTA kernel; the
 *   results are the same bit for bit. The environment variable
 *   MOE_GEMM_CTA_PAIRS, read here, overrides the choice: n > 0 takes the
 *   two-SM kernel with at most n pairs for every call, 0 the one-CTA kernel.
 *   Returns MOE_ERR_CUDA if the device is unusable.
 * moe_ctx_destroy: frees the context (NULL is ignored).
 * moe_get_device_error: synchronises `stream`, reads the error word into
 *   *bits (host) and clears it. */
MOE_API int moe_ctx_create(moe_ctx** out, int device);
MOE_API int moe_ctx_destroy(moe_ctx* ctx);
MOE_API int moe_get_device_error(moe_ctx* ctx, uint32_t* bits, moe_stream_t stream);
MOE_API const char* moe_status_string(int status);
MOE_API int moe_version(void);

/* ---------------------------------------------------- endpoints alone
 * expert_ends[e] from per-expert live-row counts[e] (both int32 [E], device):
 * start[0] = 0, start[e] = align_up(end[e-1], A), end[e] = start[e] + count[e]
 * ([LR] §2, "概念伪代码"). One block; 1 <= E <= 8192. */
MOE_API int moe_expert_ends_from_counts(moe_ctx* ctx, const int32_t* counts, int E, int A,
                                        int32_t* expert_ends, moe_stream_t stream);

/* The activation between the GEMMs (moe_act_quant, moe_grouped_gemm_act_quant,
 * moe_ffn_forward). */
typedef struct moe_act_params {
    int32_t kind;  /* MOE_ACT_* */
    float limit;   /* L for SILU_CLAMP: > 0 (+inf allowed); other values are
                      rejected with MOE_ERR_INVALID_ARG. Gate: min(g, L), up:
                      clamp(u, -L, L), a NaN operand of min / max yielding the
                      other one (IEEE minNum / maxNum). */
    float situ_beta_s; /* SITU: beta_s of the gate half (Kimi: 4), > 0, finite */
    float situ_beta_l; /* SITU: beta_l of the up half (Kimi: 25), > 0, finite.
                          SiTU ([DG] §2.4.1 situ branch, [KM] reference
                          formula; the pages print tan in the formula and tanh
                          in the code, tanh is taken): gate' = (bs tanh(g/bs))
                          sigmoid(g), up' = bl tanh(u/bl), h = gate' up', with
                          the library's exp and tanh definitions. The context
                          keeps the two 65,536-entry tables of one (bs, bl)
                          pair and refills them on the call's stream when a
                          call asks for another pair, so calls with different
                          pairs must not overlap on different streams. */
    int32_t quant_group; /* group of the e4m3 result: 128 (also 0), or 32 for
                            the MXFP8 recipe ([DG] §6): out_sf is then
                            [I/128][align4(rows)], four group-32 bytes a word */
} moe_act_params;

/* ------------------------------------------------------ route + scatter
 * [LR] §2 ("scatter 在现有步骤内写出 int32 endpoint"), [DG] §2.2.4 (compact
 * layout: per-token-group quantisation then ep_scatter into expert
 * segments), [DG] 附录 C (ep_scatter, src2dst).
 *
 * 1. Routing (unless PRECOMPUTED): per token, the k experts with the largest
 *    score, ties to the lower expert index, in descending order.
 *    SOFTMAX_TOPK: score = logit; weight_j = exp(l_j - l_max) / sum over the
 *    selected slots ([DG] §2.2.1). SIGMOID_BIAS_TOPK: score = sigmoid(l) +
 *    corr_bias; weight_j = sigmoid(l_j) / sum of the selected sigmoids
 *    ([KM] Phase 1, topk.py row). exp is the library's exp specification
 *    (Cody & Waite reduction plus a degree-7 Taylor series in fixed fp32
 *    steps, written out in csrc/common.cuh).
 * 2. Endpoints from the per-expert route counts (ids outside [0,E) skipped).
 * 3. Route (t, j) of expert e gets row start[e] + number of earlier routes
 *    (row-major (t, j) order) to e; src2dst[t,j] = that row, or -1.
 * 4. Each token row x[t] is quantised once (group 128, UE8M0, e4m3) and its
 *    codes/scales copied to each of its rows of a_fp8 / a_sf.
 *
 * Arguments (device pointers):
 *  logits [T,E] fp32 (ignored if PRECOMPUTED); corr_bias [E] fp32
 *  (SIGMOID_BIAS only, else NULL); topk_ids [T,k] int32 (written; read if
 *  PRECOMPUTED); topk_w [T,k] fp32 (written; ignored if PRECOMPUTED);
 *  x [T,H] bf16; a_fp8 [cap,H] e4m3; a_sf ASF [ceil(H/512)][align4(cap)];
 *  expert_ends [E] int32 (written); src2dst [T,k] int32 (written);
 *  workspace: moe_route_scatter_workspace_size(T,E,k) bytes of scratch
 *  (ceil(T/64) * E int32 chunk histograms and a 4-byte completion count,
 *  rounded up to 16 bytes), 16-byte aligned, contents need not be
 *  initialised; calls that share a workspace must not overlap on the GPU.
 * Sizes: T >= 0 (T == 0 writes expert_ends = 0 and nothing else; the
 *  per-token pointers may then be NULL),
 *  1 <= E <= 4096 (E <= 1024 for the two routing modes), 1 <= k <= min(E, 32),
 *  H % 128 == 0, H <= 28,160 (the scatter quantises each token row into
 *  shared memory first; larger H: MOE_ERR_UNSUPPORTED), A >= 1,
 *  cap >= T*k + E*(A-1). Logits must be finite.
 * Errors: MOE_ERR_INVALID_ARG (null pointer, bad size), MOE_ERR_CAPACITY
 *  (cap below the bound above), MOE_ERR_UNSUPPORTED (H above the limit).
 * Launches: routing, rank/count (+ endpoints), scatter; the scatter starts
 *  while rank/count still runs (programmatic dependent launch) and waits for
 *  it before it reads anything rank/count writes. */
typedef struct moe_route_args {
    int32_t routing_mode;
    const float* logits;
    const float* corr_bias;
    int32_t* topk_ids;
    float* topk_w;
    const uint16_t* x;
    uint8_t* a_fp8;
    int32_t* a_sf;
    int32_t* expert_ends;
    int32_t* src2dst;
    void* workspace;
    size_t workspace_bytes;
    int32_t T, E, k, H, A, cap;
    int32_t quant_group; /* input quantisation group: 128 (also 0), or 32 for
                            the MXFP8 recipe ([DG] §6); a_sf then holds
                            the four group-32 scale bytes of each 128 columns
                            in one word: [H/128][align4(cap)] */
} moe_route_args;

MOE_API size_t moe_route_scatter_workspace_size(int T, int E, int k);
MOE_API int moe_route_scatter(moe_ctx* ctx, const moe_route_args* args, moe_stream_t stream);

/* -------------------------------------------- route + scatter, no allocation
 * The pages have no counterpart of this entry point.
 *
 * For callers that cannot allocate device memory: code that runs inside a
 * host framework which plans and owns every device buffer and hands the
 * library only the tensors of the operation, or code on a latency-critical
 * path where an allocation (which may synchronise the device) is not allowed.
 * They cannot provide the scratch workspace moe_route_scatter needs.
 *
 * Same operation, arguments, results and errors as moe_route_scatter, except
 * that args->workspace and args->workspace_bytes are ignored: the scratch (the
 * per-chunk expert histograms, ceil(T/64) * E int32, and a 4-byte completion
 * count) lives in a device array of 1 MiB + 16 bytes inside the library.
 * Limit: ceil(T/64) * E * 4 <= 1 MiB (T <= 4096 with
 * any E <= 4096; T = 65536 with E <= 256); larger sizes return
 * MOE_ERR_UNSUPPORTED. The call allocates nothing.
 *
 * The array belongs to the library's device code: it comes into being on a
 * GPU when that code is loaded there. moe_ctx_create loads it and looks up the
 * array's device address on the context's device (cudaGetSymbolAddress), so
 * the array exists from the context's creation on and stays until the process
 * exits; this entry point itself does no set-up. All calls share the one
 * array: calls that may overlap on the GPU (on different streams, or from
 * different threads, without ordering between them) race and give wrong
 * results; order them. Nothing in the array needs clearing between calls:
 * each call writes every histogram entry before reading it, and zeroes the
 * completion count before the launch that counts in it. */
MOE_API int moe_route_scatter_noalloc(moe_ctx* ctx, const moe_route_args* args, moe_stream_t stream);

/* ------------------------------------------------------- weight prepare
 * Load-time (not on the hot path) re-layout of MXFP4 weights for the grouped
 * GEMM ([DG] §2.1.2 path A: weight scales are transformed once at load into
 * the layout the GEMM consumes). Input: packed e2m1 w_in [E][N][K/2] and
 * canonical UE8M0 bytes sf_in [E][N][K/32]. Output scales: uint32 words
 * sf_out [E][K/128][N]; the word of (e, c, n) holds the four scales of
 * k-blocks 4c..4c+3 of row n, block 4c in the low byte, and within each block
 * of 128 rows position 4i + j holds row 32j + i (the tensor-memory scale
 * layout the GEMM copies as is). Output weights w_out:
 *   MOE_GEMM_W_E2M1: packed e2m1 [E][N][K/2] (a copy; w_out may equal w_in)
 *   MOE_GEMM_W_E4M3: the same values re-encoded exactly as e4m3 [E][N][K]
 *                    (twice the bytes; [DG] §2.1.2 path B does the same
 *                    lossless widening of e2m1 to e4m3)
 * The flag MOE_GEMM_W_GATEUP_BLOCK128 (for w13 = [gate; up] halves, N = 2I)
 * also reorders the rows (and their scales) so that output rows 256b..256b+127
 * are gate rows 128b..128b+127 and rows 256b+128..256b+255 are up rows
 * I+128b..: every 256-column GEMM tile then holds one matching gate/up group,
 * which lets moe_ffn_forward run SiLU*mul and the quantisation inside GEMM1.
 * FP8 weights ([DG] §6 recipes) are prepared with the output
 * format MOE_GEMM_W_E4M3 and the input flag MOE_GEMM_W_IN_E4M3: w_in is
 * e4m3 [E][N][K] and is copied (rows reordered with the gate/up flag). Their
 * scales are per (row, 32-K) bytes [E][N][K/32] (MXFP8 recipe), or, with the
 * input flag MOE_GEMM_W_SF_BLOCK128, one UE8M0 byte per 128 x 128 block,
 * [E][ceil(N/128)][K/128] (FP8 block128 recipe), given to every 32-K slot of
 * the block. The two input flags are for this call only; the GEMMs take the
 * format without them.
 * Requires K % 128 == 0, N % 128 == 0 (N % 256 with the flag); w_out must not
 * overlap sf_out, and must differ from w_in when widening or reordering. */
#define MOE_GEMM_W_E2M1 0
#define MOE_GEMM_W_E4M3 1
#define MOE_GEMM_W_GATEUP_BLOCK128 2 /* flag, or-ed with the format: w13 only */
#define MOE_GEMM_W_IN_E4M3 4         /* moe_prepare_weights input flag: w_in is e4m3 [E][N][K] */
#define MOE_GEMM_W_SF_BLOCK128 8     /* moe_prepare_weights input flag: 128 x 128 block scales */
#define MOE_GEMM_A_GROUP32 16        /* GEMM flag: the A scales are group-32 words (MXFP8 recipe) */
MOE_API int moe_prepare_weights(moe_ctx* ctx, const uint8_t* w_in, const uint8_t* sf_in, int E, int N,
                                int K, int w_format, uint8_t* w_out, uint32_t* sf_out,
                                moe_stream_t stream);

/* ------------------------------------------------------- grouped GEMM
 * One block-scaled grouped GEMM over live rows ([LR] §2: FC1/FC2 take the
 * endpoint layout; [DG] §2.3.1, recipes (1,128) for the e4m3 activations and
 * (1,32) for the MXFP4 weights):
 *   out[r, n] = bf16( sum_k e4m3(a[r,k]) 2^(sa(r,k/128)-127)
 *                           * e2m1(w[e,n,k]) 2^(sw(e,n,k/32)-127) )
 * for r in [start[e], expert_ends[e]) only; fp32 accumulation in tensor
 * memory (tcgen05, sm_103a). a [cap,K] e4m3; a_sf ASF [ceil(K/512)][ld_sf],
 * or with the flag MOE_GEMM_A_GROUP32 in w_format (MXFP8 recipe, [DG] §6:
 * sa(r, k/32)) [K/128][ld_sf], four group-32 bytes per word;
 * w, w_sf prepared by moe_prepare_weights in format w_format ([E][N][K/2]
 * packed e2m1 or [E][N][K] e4m3; scales [E][K/128][N]); out [cap,N] bf16.
 * Requires 1 <= E <= 4096, K % 128 == 0, N % 256 == 0, cap % 128 == 0,
 * A == 128, ld_sf >= cap, ld_sf % 4 == 0, 32-byte aligned w, 16-byte
 * aligned a, a_sf, w_sf and out. */
MOE_API int moe_grouped_gemm(moe_ctx* ctx, const uint8_t* a, const int32_t* a_sf, int ld_sf,
                             const int32_t* expert_ends, int E, int A, int cap, const uint8_t* w,
                             const uint32_t* w_sf, int w_format, int N, int K, uint16_t* out,
                             moe_stream_t stream);

/* ------------------------------------- GEMM1 fused with SiLU*mul + quant
 * GEMM1 of the live rows with the activation step in its epilogue: the
 * operation of moe_grouped_gemm with w13 (N = 2I) prepared with
 * MOE_GEMM_W_GATEUP_BLOCK128, followed by that of moe_act_quant on the
 * bf16 gate/up values, without storing them ([DG] §2.4.1 fuses activation
 * and quantisation to avoid a round trip of the intermediate; here the round
 * trip of the GEMM1 output disappears too). Output: out_fp8 [cap, I] e4m3 and
 * out_sf ASF [ceil(I/512)][align4(cap)], live rows only, bitwise equal to
 * moe_grouped_gemm + moe_act_quant on the same inputs. Requires I % 128 == 0
 * and the constraints of moe_grouped_gemm (K = H). */
MOE_API int moe_grouped_gemm_act_quant(moe_ctx* ctx, const uint8_t* a, const int32_t* a_sf, int ld_sf,
                                       const int32_t* expert_ends, int E, int A, int cap, const uint8_t* w13,
                                       const uint32_t* w13_sf, int w_format, int I, int K,
                                       const moe_act_params* act, uint8_t* out_fp8, int32_t* out_sf,
                                       moe_stream_t stream);

/* ---------------------------------------------------- activation quant
 * [LR] §2-3 (live-row activation kernel: 3-D grid with the expert on axis z,
 * grid-stride loop over [start[e], end[e]), padding left unwritten; a dense
 * launch over all rows when no endpoints are given), [DG] §2.4.1 (fused
 * SiLU*mul + per-token-group quant, UE8M0 packed MN-major output;
 * silu_mul_keep_fp32: SiLU result kept in fp32).
 *   gate = gateup[r, j], up = gateup[r, I + j]
 *   SILU_CLAMP: gate = min(gate, L), up = clamp(up, -L, L) ([DG] §2.4.1)
 *   h = silu(gate) * up in fp32 (silu(g) = g / (1 + exp(-g)), the library's
 *   exp specification); per 128 columns: amax, b = ceil_pow2(amax / 448),
 *   code = e4m3_rne_satfinite(h * 2^(127-b)); amax infinite -> b = 0xFE.
 * gateup [M_alloc, 2I] bf16; out [M_alloc, I] e4m3; out_sf ASF
 * [ceil(I/512)][align4(M_alloc)]; expert_ends [E] or NULL (dense fallback:
 * every row of [0, M_alloc)). Requires I % 128 == 0, A >= 1. */


MOE_API int moe_act_quant(moe_ctx* ctx, const uint16_t* gateup, uint8_t* out, int32_t* out_sf,
                          const int32_t* expert_ends, int E, int A, int M_alloc, int I,
                          const moe_act_params* act, moe_stream_t stream);

/* ------------------------------------------------------------- combine
 * [DG] §2.6.1 (post_reorder): out[t] = bf16( rsf * sum over j = 0..k-1 with
 * src2dst[t,j] >= 0 of topk_w[t,j] * down[src2dst[t,j]] ), accumulated in
 * fp32, one fused multiply-add per slot in slot order. down [rows,H] bf16
 * (rows referenced by src2dst only); topk_w/src2dst [T,k]; out [T,H] bf16.
 * Requires H % 8 == 0. */
MOE_API int moe_combine(moe_ctx* ctx, const uint16_t* down, int H, const float* topk_w,
                        const int32_t* src2dst, int T, int k, float rsf, uint16_t* out,
                        moe_stream_t stream);

/* ----------------------------------------------------------- FFN forward
 * GEMM1 -> act-quant -> GEMM2 -> combine on one stream, all driven by the
 * device-side expert_ends ([LR] §2 "FC1(endpoint) → SiLU+mul+quant(endpoint)
 * → FC2(endpoint)"). When w13 was prepared with MOE_GEMM_W_GATEUP_BLOCK128
 * (w_format carries the flag), SiLU*mul and the quantisation run in GEMM1's
 * epilogue on its bf16-rounded accumulators, bitwise equal to the separate
 * act-quant step, and `gateup` is not used (may be NULL). Inputs: a_fp8/a_sf/expert_ends/src2dst as written by
 * moe_route_scatter; topk_w [T,k]; w13 [E][2I][H/2] and w2 [E][H][I/2]
 * prepared with their scales by moe_prepare_weights. Workspaces (caller
 * owned, fixed capacity, contents need not be initialised): gateup
 * [cap,2I] bf16, act_fp8 [cap,I], act_sf ASF [ceil(I/512)][align4(cap)],
 * down [cap,H] bf16. Output out [T,H] bf16. Requires H % 256 == 0,
 * I % 128 == 0, 2I % 256 == 0, A == 128, cap % 128 == 0. */
typedef struct moe_ffn_args {
    const uint8_t* a_fp8;
    const int32_t* a_sf;
    const int32_t* expert_ends;
    const uint8_t* w13;
    const uint32_t* w13_sf;
    const uint8_t* w2;
    const uint32_t* w2_sf;
    uint16_t* gateup;
    uint8_t* act_fp8;
    int32_t* act_sf;
    uint16_t* down;
    const float* topk_w;
    const int32_t* src2dst;
    uint16_t* out;
    int32_t T, E, k, H, I, A, cap;
    int32_t w_format; /* MOE_GEMM_W_*, the format both w13 and w2 were prepared in */
    moe_act_params act;
    float rsf;
} moe_ffn_args;

MOE_API int moe_ffn_forward(moe_ctx* ctx, const moe_ffn_args* args, moe_stream_t stream);

/* ------------------------------------------------ sparse decode GEMV
 * [SD] §3: per (token, slot) whose expert e is local (expert_start <= e <
 * expert_start + num_local_experts), block-uniformly read from topk_ids on
 * the device:
 *   y1[t,j] = W_gu[e] x[t] (* scale) + b_gu[e]            bf16 [T,k,2I]
 *   act[t*k+j] = GLU(y1[t,j])                             bf16 [T*k, I]
 *   y2[t,j] = W_d[e] act[t*k+j] (* scale) + b_d[e]        bf16 [T,k,H]
 *   out[t] = bf16( sum over local slots, in slot order, of topk_w * y2 )
 * Slots of non-local experts are never written and are skipped in the sum,
 * never multiplied by zero ([SD] §3 "两个容易写错的安全点").
 * GLU: g = min(g, L), u = clamp(u, -L, L) (L <= 0: no clamp),
 *   act = (g * sigmoid(alpha g)) * (u + beta); layout HALVES or INTERLEAVED.
 * Weights (local expert index lid = e - expert_start):
 *   FP8_PER_EXPERT: w_gu [n_local][2I][H] e4m3, w_gu_scale [n_local] fp32,
 *                   w_d [n_local][H][I], w_d_scale [n_local]
 *   MXFP4_G32:      w_gu [n_local][2I][H/2], w_gu_sf [n_local][2I][H/32],
 *                   w_d [n_local][H][I/2], w_d_sf [n_local][H][I/32]
 *   b_gu [n_local][2I] bf16, b_d [n_local][H] bf16.
 * Requires H % 32 == 0, I % 32 == 0, k <= 32, and T <= 64 -- or T <= 128
 * with a workspace; w_gu, w_d, the MXFP4 scale arrays and the biases 16-byte
 * aligned, x and act 8-byte aligned. y1 / y2 / act of non-local slots are
 * never written.
 * Paths (args.path; AUTO takes the tcgen05 path when it applies and T >= 8
 * for FP8 or T >= 4 for MXFP4 -- below that the mma.sync path is faster,
 * when it applies --, else the mma.sync path, else the GEMV path; a forced
 * path that does not apply is an invalid argument). The first two read every
 * selected local expert's weights once for all the slots that chose it
 * ([SD] §4 crossover removed):
 *   - TCGEN05: workspace given (at least moe_decode_workspace_size() bytes, 256-byte
 *     aligned, owned by the caller, contents need not be initialised; not
 *     shared by calls in flight at the same time), T * k <= 4096,
 *     num_local_experts <= 1024, H, I >= 128, and for MXFP4 H, I <= 4096,
 *     H % 64 == I % 64 == 0 and w_gu, w_d 32-byte aligned, y1, act, y2
 *     16-byte aligned: the tcgen05
 *     block-scaled path. The slots are grouped by expert into 16-row
 *     aligned segments; each bf16 activation row (x, then act) is fed to the
 *     MMA as two e4m3 terms with group-32 UE8M0 scales (hi = e4m3(v / s_hi),
 *     lo = e4m3((v - hi s_hi) / s_lo)), which reproduce every value within
 *     2^13 of its group's maximum exactly and the others to 2^-21 of that
 *     maximum; the weights enter the tensor cores in their stored format.
 *   - MMA_SYNC: T <= 8 with H % 64 == 0 and I % 64 == 0: m16n8k16 f16 MMA
 *     on exactly converted weights against token columns scaled per token by
 *     a power of two;
 *   - GEMV: one GEMV block per (token, slot, 32 rows), T <= 64. */
typedef struct moe_decode_args {
    const uint16_t* x;
    const int32_t* topk_ids;
    const float* topk_w;
    int32_t expert_start, num_local_experts, wfmt;
    const uint8_t* w_gu;
    const float* w_gu_scale;
    const uint8_t* w_gu_sf;
    const uint16_t* b_gu;
    const uint8_t* w_d;
    const float* w_d_scale;
    const uint8_t* w_d_sf;
    const uint16_t* b_d;
    int32_t glu_layout;
    float glu_alpha, glu_beta, glu_limit;
    uint16_t* y1;
    uint16_t* act;
    uint16_t* y2;
    uint16_t* out;
    int32_t T, H, I, k;
    void* workspace;        /* device scratch of the tcgen05 path, or NULL */
    size_t workspace_bytes;
    int32_t path;           /* MOE_DECODE_* */
} moe_decode_args;

/* Bytes of the tcgen05 decode path's workspace for these sizes (0 when the
 * sizes are out of range). */
MOE_API size_t moe_decode_workspace_size(int32_t T, int32_t k, int32_t H, int32_t I, int32_t num_local_experts);
MOE_API int moe_sparse_gemv_decode(moe_ctx* ctx, const moe_decode_args* args, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
