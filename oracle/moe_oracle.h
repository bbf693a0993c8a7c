/*
 * moe_oracle.h -- declarations of the CPU oracle for the routed MoE expert FFN.
 *
 * TEST INFRASTRUCTURE ONLY. The oracle is a plain, slow, obviously correct CPU
 * restatement of what the hot path computes. Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg load it; the CUDA library never
 * includes this header, never links this code and shares no helper with it.
 *
 * Parity partly unpinned (see the per-function notes):
 *   - orc_glu_oai: the gpt-oss GLU of the decode path; its clamp and the
 *     place of alpha are pinned, the place of beta is a reading.
 *
 * Conventions
 *   bf16 values travel as uint16_t bit patterns; fp8-e4m3 codes as uint8_t;
 *   packed e2m1 as uint8_t with the LOW nibble holding the even K index;
 *   UE8M0 scales as uint8_t exponent bytes (value 2^(b-127)).
 *   Packed activation scales: int32 array [ceil(G/4)][ld] ("MN-major"), where
 *   byte (g % 4) of word [g/4][row] is the scale of 128-column group g.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* number formats */
float    orc_bf16_to_float(uint16_t h);
uint16_t orc_bf16_from_float(float f);
uint16_t orc_bf16_from_double(double d);
double   orc_e4m3_value(uint8_t code);
uint8_t  orc_e4m3_from_float(float x);
double   orc_e2m1_value(uint8_t nibble);
double   orc_ue8m0_value(uint8_t b);
uint8_t  orc_ue8m0_ceil(float s);

/* the exp / SiLU / sigmoid specification shared by both sides of the check */
float orc_exp_spec(float x);
float orc_silu_spec(float g);
float orc_sigmoid_spec(float x);
float orc_tanh_spec(float y);
float orc_situ_gate_spec(float g, float beta_s);
float orc_situ_up_spec(float u, float beta_l);

/* activation between the GEMMs: kind 0 SiLU, 1 SiLU with clamp limit,
 * 2 SiTU with beta_s (gate) and beta_l (up) */
typedef struct orc_act {
    int kind;
    float limit, beta_s, beta_l;
    int group; /* quantisation group of the result: 128, or 32 (MXFP8 recipe) */
} orc_act;

/* group-128 e4m3 quantisation of one fp32 row */
void orc_group_quant_row(const float* v, int K, int group, uint8_t* codes, uint8_t* scales);

/* routing */
void orc_route_softmax_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w);
void orc_route_sigmoid_bias_topk(const float* logits, const float* bias, int T, int E, int k,
                                 int32_t* ids, float* w);

/* endpoints and scatter */
void orc_expert_counts(const int32_t* ids, long R, int E, int32_t* counts);
void orc_endpoints(const int32_t* counts, int E, int A, int32_t* start, int32_t* end);
int  orc_scatter(const int32_t* ids, const uint16_t* x, int T, int k, int E, int H, int A, int cap,
                 int ld_sf, int group, int32_t* expert_ends, int32_t* src2dst, uint8_t* a_fp8, int32_t* a_sf);

/* grouped block-scaled GEMM over live rows (fp64 accumulation, one bf16
 * rounding); a_group 128 or 32; wfmt 0 packed e2m1 [E][N][K/2], 1 e4m3 [E][N][K];
 * weight scales per (row, 32-K) bytes [E][N][K/32] */
void orc_grouped_gemm(const uint8_t* a, const int32_t* a_sf, int ld_sf, int K, int a_group,
                      const int32_t* expert_ends, int E, int A,
                      const uint8_t* w, const uint8_t* w_sf, int wfmt, int N, uint16_t* out);
void orc_expand_block_scales(const uint8_t* sf_blk, int E, int N, int K, uint8_t* sf32);

/* live-row SiLU*mul + e4m3/UE8M0 quantisation; expert_ends == NULL means every row */
void orc_act_quant(const uint16_t* gateup, int M_alloc, int I, const int32_t* expert_ends, int E,
                   int A, int act_kind, float limit, float beta_s, float beta_l, int group, uint8_t* out,
                   int32_t* out_sf, int ld_sf);

/* top-k weighted combine */
void orc_combine(const uint16_t* down, int H, const float* topk_w, const int32_t* src2dst, int T,
                 int k, float rsf, uint16_t* out);

/* whole layer, per token, computing only the selected experts (used for samples) */
void orc_ffn_tokens(const uint16_t* x, int H, int I, const int32_t* ids, const float* topk_w, int k,
                    int E, const uint8_t* w13, const uint8_t* w13_sf, const uint8_t* w2,
                    const uint8_t* w2_sf, int wfmt, int group, int act_kind, float limit, float beta_s,
                    float beta_l, float rsf, const int32_t* tokens, int n_tokens, uint16_t* out);

/* dense twin: every expert on every token, then select by routing and sum */
void orc_ffn_dense(const uint16_t* x, int T, int H, int I, const int32_t* ids, const float* topk_w,
                   int k, int E, const uint8_t* w13, const uint8_t* w13_sf, const uint8_t* w2,
                   const uint8_t* w2_sf, int wfmt, int group, int act_kind, float limit, float beta_s,
                   float beta_l, float rsf, uint16_t* out);

/* decode GEMV path (bf16 activations, FP8-per-expert or MXFP4 weights) */
float orc_glu_oai(float g, float u, float alpha, float beta, float limit);
void orc_decode_gemv1(const uint16_t* x, int T, int H, int I, const int32_t* ids, int k, int expert_start,
                      int n_local, int wfmt, const uint8_t* w_gu, const float* gu_scale, const uint8_t* gu_sf,
                      const uint16_t* b_gu, uint16_t* y1);
void orc_decode_glu(const uint16_t* y1, int T, int I, const int32_t* ids, int k, int expert_start, int n_local,
                    int glu_interleaved, float alpha, float beta, float limit, uint16_t* act);
void orc_decode_gemv2(const uint16_t* act, int T, int H, int I, const int32_t* ids, int k, int expert_start,
                      int n_local, int wfmt, const uint8_t* w_d, const float* d_scale, const uint8_t* d_sf,
                      const uint16_t* b_d, uint16_t* y2);
void orc_decode_sum(const uint16_t* y2, int T, int H, const int32_t* ids, const float* topk_w, int k,
                    int expert_start, int n_local, uint16_t* out);
void orc_decode(const uint16_t* x, int T, int H, int I, const int32_t* ids, const float* topk_w, int k,
                int expert_start, int n_local, int wfmt,
                const uint8_t* w_gu, const float* gu_scale, const uint8_t* gu_sf, const uint16_t* b_gu,
                const uint8_t* w_d, const float* d_scale, const uint8_t* d_sf, const uint16_t* b_d,
                int glu_interleaved, float alpha, float beta, float limit,
                uint16_t* y1, uint16_t* act, uint16_t* y2, uint16_t* out);
void orc_decode_dense(const uint16_t* x, int T, int H, int I, const int32_t* ids, const float* topk_w,
                      int k, int expert_start, int n_local, int wfmt,
                      const uint8_t* w_gu, const float* gu_scale, const uint8_t* gu_sf,
                      const uint16_t* b_gu, const uint8_t* w_d, const float* d_scale,
                      const uint8_t* d_sf, const uint16_t* b_d, int glu_interleaved, float alpha,
                      float beta, float limit, uint16_t* out);

int orc_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
