/*
 * mx_oracle.h -- plain, slow CPU oracle for the block-scaled (microscaling)
 * low-precision linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this code: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library; it has its own enums below.
 *
 * Sources (web pages; cited by title and section):
 *   [MOSS]  "MOSS: 用微缩放和自动缩放实现无损 FP8 训练，OLMo-7B 加速 34%"
 *           sections 创新 1 (two-level figure), Power-of-Two 的关键优势,
 *           两级缩放实现 (TwoLevelMicroScaling), GEMM Kernel 优化.
 *   [COAT]  "COAT: Compressing Optimizer States and Activation for memory
 *           efficient FP8 Training" (article), section FP8 量化最佳化器狀態的難點.
 *   [FAF]   "格式感知融合:让FP4预训练提速两倍的工程实践", sections
 *           FP4加速为何常常"纸上富贵", 格式感知融合的设计思路, 两个关键的数值技巧.
 */
#ifndef MX_ORACLE_H
#define MX_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Oracle-private enums (deliberately separate from the library's). */
enum { ORC_FMT_MXFP8 = 0, ORC_FMT_MXFP4 = 1, ORC_FMT_NVFP4 = 2, ORC_FMT_MOSS = 3, ORC_FMT_NVFP4_LOCAL = 4 };
/* Rows of the K-major operand that share one FP32 scale in ORC_FMT_NVFP4_LOCAL. */
enum { ORC_LOCAL_REGION = 128 };
enum { ORC_ROUND_RNE = 0, ORC_ROUND_SR = 1 };
enum { ORC_RULE_DEFAULT = 0, ORC_RULE_FLOOR = 1, ORC_RULE_CEIL = 2, ORC_RULE_NEAREST = 3 };
enum { ORC_ROWWISE = 0, ORC_COLWISE = 1 };
enum { ORC_ELEM_E4M3 = 0, ORC_ELEM_E2M1 = 1 };
enum { ORC_OK = 0, ORC_ERR_ARG = 1, ORC_ERR_UNSUPPORTED = 2 };

float    orc_bf16_to_f32(uint16_t h);
uint16_t orc_f32_to_bf16_rne(float f);

double   orc_decode_e4m3(unsigned code);
double   orc_decode_e2m1(unsigned code);
double   orc_decode_e8m0(unsigned code);
unsigned orc_encode_e4m3_rne(float v);
unsigned orc_encode_e2m1_rne(float v);
unsigned orc_encode_e2m1_sr(float v, unsigned u16);
unsigned orc_encode_e4m3_sr(float v, unsigned u16);
int      orc_pow2_exponent(float block_amax, int rule, int elem);

void     orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
unsigned orc_sr_u16(uint64_t seed, uint32_t stream_id, uint64_t L);
void     orc_fwht32(float x[32]);

int64_t  orc_sf_index(int64_t r, int64_t kb, int64_t kblocks);
int64_t  orc_sf_bytes(int64_t rows, int64_t kblocks);
void     orc_sf_swizzle(const uint8_t* sf_logical, int64_t rows, int64_t kblocks, uint8_t* out);

float    orc_amax_bf16(const uint16_t* x, int64_t R, int64_t C, int64_t ld);
int      orc_quantize(const uint16_t* x, int64_t R, int64_t C, int64_t ld, int dir, int fmt,
                      int block, int rounding, int rule, uint64_t seed, uint32_t stream_id,
                      int hadamard, const float* amax_in, uint8_t* codes, uint8_t* sf_logical,
                      float* amax_out, float* tensor_scale_out);
int      orc_quantize_rows_f32(const float* x, int64_t R, int64_t C, int64_t ld, int fmt,
                               uint8_t* codes, uint8_t* sf_logical);
void     orc_dequantize(const uint8_t* codes, const uint8_t* sf_logical, int64_t rows, int64_t k,
                        int fmt, int block, double* out);
float    orc_gemm_alpha(const float* ts_a, const float* ts_b, float extra);
void     orc_gemm_q(const uint8_t* a_codes, const uint8_t* a_sf, const uint8_t* b_codes,
                    const uint8_t* b_sf, int fmt, int block, int64_t M, int64_t N, int64_t K,
                    double alpha, const int64_t* rows, int64_t nrows, const int64_t* cols,
                    int64_t ncols, double* C, double* Cabs);
int      orc_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
