/*
 * oracle.h — plain CPU reference of the routed-MoE block.  TEST
 * INFRASTRUCTURE ONLY: it is called by tests/, the smoke check and the CPU
 * baseline leg of bench.py, never by the library.  It shares no code with the
 * CUDA path and takes the blocks in their GGUF format (not the packed device
 * layout), so packing mistakes cannot cancel out.
 *
 * Every function is the plain definition written out: fp32 dequantisation in
 * the canonical order, then fp64 accumulation, full sorts, no blocking.
 * Dimensions are parameters so tiny cases can be brute-forced; the GPU path
 * only supports H = 4096, F = 2048, E = 256, K = 6.
 *
 * Sources: [P5] juejin.cn "Redis 作者出手！ds4：用 C 语言从零打造 DeepSeek V4
 * Flash 本地推理引擎" §2.1 (dims), §2.3 (block structs), §2.4 (grid rows of 8
 * int8); [P1] chenxutan.com "ds4 深度实战" §2.1 (which tensors are 2-bit), §3.2
 * (moe_forward steps).  Readings where the pages are silent are listed at each
 * function.
 *
 * Parity status: real-model numerics (the real IQ2_XXS codebook, trained
 * weights) are unpinned — no table, weights or vectors are available; the
 * codebook is a seeded stand-in passed as data.
 */
#ifndef DS4_ORACLE_H
#define DS4_ORACLE_H
#include <stddef.h>
#include <stdint.h>

#define ORACLE_IQ2_XXS 0
#define ORACLE_Q2_K 1
#define ORACLE_Q4_K 2
#define ORACLE_BF16 3

/* fp16 bits -> fp32, exact (subnormals, inf, nan). */
float oracle_fp16_to_f32(uint16_t h);
/* fp32 -> bf16 bits, round to nearest even (nan stays nan). */
uint16_t oracle_f32_to_bf16(float f);
/* GGUF block size in bytes for a type (66, 84, 144), 0 otherwise. */
int oracle_block_bytes(int qtype);

/* Dequantise one row of cols/256 GGUF blocks to fp32.  grid: 256 x 8 uint8
 * (IQ2_XXS only).  Returns 0, or -1 on a bad argument. */
int oracle_dequant_row(int qtype, const uint8_t *row_blocks, int cols,
                       const uint8_t *grid, float *out);
/* Whole matrix; out_f32 and/or out_bf16 may be NULL. */
int oracle_dequantize(int qtype, const void *gguf, int rows, int cols,
                      const uint8_t *grid, float *out_f32, uint16_t *out_bf16);

/* Router for T tokens.  keys_out [T][E] (may be NULL) receives s_e + bias_e,
 * margin_out [T] (may be NULL) receives key of the K-th pick minus key of the
 * (K+1)-th (the distance to the nearest routing flip). */
int oracle_route(const float *hidden, int T, int H, int E, int K,
                 const float *router, const float *bias, int32_t *ids,
                 float *w, double *keys_out, double *margin_out);

/* Counting sort of the T*K entries by expert, stable in (t,k) order. */
int oracle_bucket(const int32_t *ids, int T, int K, int E, int32_t *counts,
                  int32_t *offsets, int32_t *perm, int32_t *inv);

/* y = x / sqrt(mean(x^2) + eps), per row of n. */
void oracle_rmsnorm(const float *x, int T, int n, double eps, float *y);

/* The MoE block for T tokens given ids/w.  gate/up/down: arrays of E
 * pointers to GGUF-format matrices (gate/up [F][H], down [H][F]); entries for
 * experts no token selects may be NULL.  sh_*: bf16 bits, row-major.  out
 * [T][H].  nthreads <= 0 means the OpenMP default.  Returns 0, -1 on a bad
 * argument, -2 on an id outside [0,E) or a missing expert. */
int oracle_moe_forward(const float *hidden, int T, int H, int F, int E, int K,
                       int gate_up_type, int down_type,
                       const void *const *gate, const void *const *up,
                       const void *const *down, const uint16_t *sh_gate,
                       const uint16_t *sh_up, const uint16_t *sh_down,
                       const uint8_t *grid, const int32_t *ids, const float *w,
                       float *out, int nthreads);

/* One expert's MLP for one token: y = D (silu(G x) * (U x)), fp64 out [H].
 * qtype ORACLE_BF16 means a row-major bf16 matrix. */
int oracle_expert_mlp(const float *x, int H, int F, int gate_up_type,
                      int down_type, const void *G, const void *U,
                      const void *D, const uint8_t *grid, double *y,
                      int nthreads);

/* q8 activations (the int8 path: chenxutan ds4 article §2.4, the
 * dot_iq2_pair_16 kernel, int8 grid values against int8 activations).
 * Reading (the pages give the dot, not the quantiser): blocks of 256
 * columns; d = max|x| / 127 in fp32 (0 for an all-zero block); q = x / d in
 * fp32 rounded to the nearest integer, ties to even, clamped to [-127, 127].
 * q [n] int8, d [n / 256]; n a multiple of 256.  Returns 0 or -1. */
int oracle_quantize_q8(const float *x, int n, int8_t *q, float *d);

/* oracle_moe_forward with the routed IQ2_XXS gate and up projections on q8
 * activations: per 32-weight sub-block the exact integer sum S of
 * (sign * grid value) * q (as dot_iq2_pair_16 forms it, 16 products at a
 * time), then row += db * d_x * S (fp64, in index order; db the sub-block
 * scale of the format).  The down projection and the shared expert are as in
 * oracle_moe_forward.  gate_up_type must be IQ2_XXS (-1 otherwise). */
int oracle_moe_forward_q8(const float *hidden, int T, int H, int F, int E, int K,
                          int gate_up_type, int down_type,
                          const void *const *gate, const void *const *up,
                          const void *const *down, const uint16_t *sh_gate,
                          const uint16_t *sh_up, const uint16_t *sh_down,
                          const uint8_t *grid, const int32_t *ids, const float *w,
                          float *out, int nthreads);

#endif
