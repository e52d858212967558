/*
 * tfx_oracle.h -- the CPU oracle's own declarations (test infrastructure only; see
 * tfx_oracle.c). Nothing here is shared with the CUDA library.
 */
#ifndef TFX_ORACLE_H
#define TFX_ORACLE_H
#include <stdint.h>

#define TFXO_ACT_E4M3 0
#define TFXO_ACT_BF16 1

#define TFXO_ST_RANGE 1
#define TFXO_ST_DUP 2

double tfxo_e2m1_value(int code);
double tfxo_e4m3_value(int code);
double tfxo_ue8m0_value(int code);
float tfxo_bf16_to_f32(uint16_t b);
uint16_t tfxo_f32_to_bf16(float f);
uint16_t tfxo_f64_to_bf16(double v);
int tfxo_e4m3_encode(double v);

void tfxo_quant_e4m3_f32(int n, const float* h, uint8_t* codes, uint8_t* scales);
void tfxo_quant_e4m3_f64(int n, const double* h, uint8_t* codes, uint8_t* scales);
void tfxo_round_bf16(int n, const float* h, uint16_t* out);
void tfxo_round_bf16_f64(int n, const double* h, uint16_t* out);

int tfxo_route(const int32_t* ids, int R, int k, int E, int32_t* offs, int32_t* pair_row,
               int32_t* pair_slot, int32_t* active, int32_t* n_active);

float tfxo_chain_dot(int K, const uint8_t* wc, const uint8_t* ws, const float* xc, const float* xs);
double tfxo_f64_dot(int K, const uint8_t* wc, const uint8_t* ws, const double* xh, double* mass);

void tfxo_gateup_chain(int H, int I, const uint8_t* wg, const uint8_t* sg, const uint8_t* wu,
                       const uint8_t* su, int kind, const void* x, const uint8_t* sx, float* xbuf,
                       float* g, float* u);
void tfxo_gateup_f64(int H, int I, const uint8_t* wg, const uint8_t* sg, const uint8_t* wu,
                     const uint8_t* su, int kind, const void* x, const uint8_t* sx, double* xbuf,
                     double* g, double* u, double* mg, double* mu);
void tfxo_silu_mul_f32(int n, const float* g, const float* u, float* h);
void tfxo_silu_mul_f64(int n, const double* g, const double* u, const double* mg, const double* mu,
                       double* h, double* mh);
void tfxo_down_chain(int H, int I, const uint8_t* wd, const uint8_t* sd, int kind, const void* h,
                     const uint8_t* sh, float* xbuf, float* d);
void tfxo_down_f64(int H, int I, const uint8_t* wd, const uint8_t* sd, int kind, const void* h,
                   const uint8_t* sh, double* xbuf, double* d, double* md);
void tfxo_combine_chain(int k, int H, const float* d, const float* w, uint16_t* y_bf16, float* y_f32);
void tfxo_combine_f64(int k, int H, const double* d, const double* md, const float* w, double* y,
                      double* my);
#endif
