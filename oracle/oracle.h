/*
 * Plain CPU oracle for the draft-head argmax path: declarations.
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
 * benchmark's CPU baseline; the product library never includes this header.
 * Every function is defined in oracle.c, which states the passage it follows.
 */
#ifndef DVL_ORACLE_H
#define DVL_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

float oracle_bf16_to_f32(uint16_t b);
float oracle_e2m1(uint8_t code);
float oracle_e4m3(uint8_t byte);
float oracle_nvfp4_weight(const uint8_t *q, const uint8_t *scales, float g, int64_t K,
                          int64_t n, int64_t k);

int oracle_num_cores(void);
int oracle_logits_bf16(const uint16_t *w, int64_t N, int64_t K, const uint16_t *h,
                       int64_t M, float *logits, int nthreads);
int oracle_logits_nvfp4(const uint8_t *q, const uint8_t *scales, float g, int64_t N,
                        int64_t K, const uint16_t *h, int64_t M, float *logits,
                        int nthreads);
int oracle_logits_fp8(const uint8_t *q, float g, int64_t N, int64_t K, const uint16_t *h,
                      int64_t M, float *logits, int nthreads);
void oracle_score_ids_fp8(const uint8_t *q, float g, int64_t N, int64_t K, int64_t id_base,
                          const uint16_t *h, int64_t M, const int32_t *ids, int64_t c,
                          float *out);
void oracle_score_ids_bf16(const uint16_t *w, int64_t N, int64_t K, int64_t id_base,
                           const uint16_t *h, int64_t M, const int32_t *ids, int64_t c,
                           float *out);
void oracle_score_ids_nvfp4(const uint8_t *q, const uint8_t *scales, float g, int64_t N,
                            int64_t K, int64_t id_base, const uint16_t *h, int64_t M,
                            const int32_t *ids, int64_t c, float *out);
float oracle_quantize_nvfp4(const uint16_t *w, int64_t N, int64_t K, uint8_t *q,
                            uint8_t *scales);
float oracle_quantize_fp8(const uint16_t *w, int64_t N, int64_t K, uint8_t *q);
void oracle_topk(const float *logits, int64_t N, int64_t M, const int32_t *d2t, int k,
                 int32_t *ids, float *vals, int64_t *rows);

int64_t oracle_check_trim(const uint8_t *w_full, int64_t V, int64_t row_bytes,
                          const int32_t *ranks, int64_t n, const uint8_t *w_trim,
                          const int32_t *d2t);

int oracle_histogram(const int32_t *tokens, int64_t n, int64_t V, int64_t *counts);
int64_t oracle_build_ranks(const int64_t *counts, int64_t V, const int32_t *forced,
                           int64_t n_forced, int64_t N, int sorted, int32_t *out);
int64_t oracle_union_sorted(const int32_t *a, int64_t na, const int32_t *b, int64_t nb,
                            int32_t *out);

#ifdef __cplusplus
}
#endif
#endif
