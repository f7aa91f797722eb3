// dequant.cu — packed tile-block layout -> fp32 / bf16 weights.  Exposes the
// exact fp32 arithmetic of the block formats (juejin ds4 article §2.3 block
// structs; inner layout per the GGUF convention) so it can be compared bit for
// bit; every product/sum below is one IEEE rounding (explicit _rn intrinsics,
// no contraction).
#include "ds4g_internal.cuh"

namespace ds4g {

__device__ __forceinline__ uint32_t ld_u32(const uint8_t *p) {
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}
__device__ __forceinline__ float ld_f16(const uint8_t *p) {
    return __half2float(__ushort_as_half((unsigned short)(p[0] | (p[1] << 8))));
}

__device__ __forceinline__ void put(float *of, uint16_t *ob, size_t idx, float w) {
    if (of) of[idx] = w;
    if (ob) ob[idx] = __bfloat16_as_ushort(__float2bfloat16_rn(w));
}

// One thread per (row, 32-weight group).
__global__ void dequant_kernel(int qt, const uint8_t *__restrict__ packed, int rows, int cols,
                               const uint64_t *__restrict__ grid, float *of, uint16_t *ob) {
    const int nb = cols / 256;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)rows * nb * 8) return;
    const int part = (int)(idx & 7);
    const long long rb = idx >> 3;
    const int r = (int)(rb / nb), b = (int)(rb % nb);
    const int rr = r & 15, g = rr & 7, hrow = rr >> 3;
    const uint8_t *tb = packed + ((size_t)(r >> 4) * nb + b) * tile_block_bytes(qt);
    const size_t obase = (size_t)r * cols + 256 * b + 32 * part;

    if (qt == DS4G_IQ2_XXS) {
        const int j = part, t = j & 3, jj = j >> 2;
        const uint8_t *rec = tb + 512 * hrow + 16 * (4 * g + t) + 8 * jj;
        const uint32_t ia = ld_u32(rec), v = ld_u32(rec + 4);
        const float d = ld_f16(tb + 1024 + 4 * g + 2 * hrow);
        const float db = __fmul_rn(__fmul_rn(d, __fadd_rn(0.5f, (float)(v >> 28))), 0.25f);
        for (int l = 0; l < 4; ++l) {
            const uint64_t row = grid[(ia >> (8 * l)) & 255u];
            const uint32_t s7 = (v >> (7 * l)) & 127u;
            const uint32_t signs = s7 | ((uint32_t)(__popc(s7) & 1) << 7);
            for (int jx = 0; jx < 8; ++jx) {
                int gv = (int)((row >> (8 * jx)) & 255u);
                if ((signs >> jx) & 1u) gv = -gv;
                put(of, ob, obase + 8 * l + jx, __fmul_rn(db, (float)gv));
            }
        }
    } else if (qt == DS4G_Q2_K) {
        const uint8_t *dd = tb + 1280 + 8 * g + 4 * hrow;
        const float d = ld_f16(dd), dmin = ld_f16(dd + 2);
        for (int k = 0; k < 32; ++k) {
            const int n = 32 * part + k;
            const int sb = n >> 4, i = n & 15, t = sb & 3, G = sb >> 2, c = i >> 2, p = i & 3;
            const uint32_t word = ld_u32(tb + 512 * hrow + 16 * (4 * g + t) + 4 * G);
            const uint32_t q = (word >> (16 * (p & 1) + 2 * (2 * c + (p >> 1)))) & 3u;
            const uint32_t scb = tb[1024 + 128 * hrow + 4 * (4 * g + t) + G];
            const float w = __fmaf_rn(__fmul_rn(d, (float)(scb & 15u)), (float)q,
                                      -__fmul_rn(dmin, (float)(scb >> 4)));
            put(of, ob, obase + k, w);
        }
    } else {  // Q4_K
        const int j = part, t = j & 3, jj = j >> 2;
        const uint8_t *s = tb + 2048 + 12 * rr;
        uint32_t sc, m;
        if (j < 4) {
            sc = s[j] & 63u;
            m = s[j + 4] & 63u;
        } else {
            sc = (s[j + 4] & 15u) | ((uint32_t)(s[j - 4] >> 6) << 4);
            m = (uint32_t)(s[j + 4] >> 4) | ((uint32_t)(s[j] >> 6) << 4);
        }
        const uint8_t *dd = tb + 2240 + 8 * g + 4 * hrow;
        const float d = ld_f16(dd), dmin = ld_f16(dd + 2);
        const float dsc = __fmul_rn(d, (float)sc), dm = __fmul_rn(dmin, (float)m);
        for (int i = 0; i < 32; ++i) {
            const int c = i >> 2, p = i & 3;
            const uint32_t word = ld_u32(tb + 1024 * hrow + 32 * (4 * g + t) + 4 * (4 * jj + (c >> 1)));
            const uint32_t q = (word >> (16 * (p & 1) + 4 * (2 * (c & 1) + (p >> 1)))) & 15u;
            put(of, ob, obase + i, __fmaf_rn(dsc, (float)q, -dm));
        }
    }
}

}  // namespace ds4g

using namespace ds4g;

extern "C" ds4g_status ds4g_dequantize(ds4g_qtype t, const void *packed, int rows, int cols,
                                       const uint64_t *iq2_grid, float *out_f32, uint16_t *out_bf16,
                                       ds4g_stream_t s) {
    DS4G_TRACE();
    if (!packed || (!out_f32 && !out_bf16)) return DS4G_EINVAL;
    if (t != DS4G_IQ2_XXS && t != DS4G_Q2_K && t != DS4G_Q4_K) return DS4G_EINVAL;
    if (t == DS4G_IQ2_XXS && !iq2_grid) return DS4G_EINVAL;
    if (rows <= 0 || cols <= 0 || rows % 16 || cols % 256) return DS4G_EUNSUPPORTED;
    if (((uintptr_t)packed | (uintptr_t)out_f32 | (uintptr_t)out_bf16 | (uintptr_t)iq2_grid) & 15)
        return DS4G_EALIGN;
    const long long n = (long long)rows * (cols / 256) * 8;
    dequant_kernel<<<(unsigned)((n + 255) / 256), 256, 0, (cudaStream_t)s>>>(
        t, (const uint8_t *)packed, rows, cols, iq2_grid, out_f32, out_bf16);
    return cudaGetLastError() == cudaSuccess ? DS4G_OK : DS4G_ECUDA;
}
