// pack.cu — GGUF-format blocks <-> packed tile-block layout (layout only: the
// bytes, 2-bit and 4-bit fields are moved, never combined arithmetically).
// The block structs are those of the juejin ds4 article, §2.3 (block_q2_K
// 84 B, block_iq2_xxs 66 B) plus the 144-byte Q4_K block of the q4 layers.
#include <string.h>

#include "ds4g_internal.cuh"

namespace ds4g {

// Move one 256-weight GGUF block of tile row rr (0..15) into / out of the
// tile-block at `tb`.  `to_packed` selects the direction.  Touches only the
// bytes of row rr, so rows and blocks can be handled in parallel.
__host__ __device__ inline void map_block(int qt, uint8_t *gguf, uint8_t *tb, int rr,
                                          bool to_packed) {
    const int g = rr & 7, hrow = rr >> 3;
    if (qt == DS4G_IQ2_XXS) {
        for (int j = 0; j < 8; ++j) {
            const int t = j & 3, jj = j >> 2;
            uint8_t *dst = tb + 512 * hrow + 16 * (4 * g + t) + 8 * jj;
            uint8_t *src = gguf + 2 + 8 * j;
            for (int i = 0; i < 8; ++i) {
                if (to_packed) dst[i] = src[i];
                else src[i] = dst[i];
            }
        }
        uint8_t *dd = tb + 1024 + 4 * g + 2 * hrow;
        for (int i = 0; i < 2; ++i) {
            if (to_packed) dd[i] = gguf[i];
            else gguf[i] = dd[i];
        }
        return;
    }
    if (qt == DS4G_Q2_K) {
        // quants: weight n = 128h + 32jq + l is field jq of qs[32h + l] (GGUF)
        uint32_t words[4][4];  // [t][G]
        for (int t = 0; t < 4; ++t)
            for (int G = 0; G < 4; ++G) {
                uint8_t *p = tb + 512 * hrow + 16 * (4 * g + t) + 4 * G;
                words[t][G] = to_packed ? 0u
                                        : (uint32_t)p[0] | ((uint32_t)p[1] << 8) |
                                              ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
            }
        uint8_t *qs = gguf + 16;
        if (!to_packed)
            for (int i = 0; i < 64; ++i) qs[i] = 0;
        for (int n = 0; n < 256; ++n) {
            const int h = n >> 7, jq = (n & 127) >> 5, l = n & 31;
            const int sb = n >> 4, i = n & 15, t = sb & 3, G = sb >> 2;
            const int c = i >> 2, p = i & 3;
            const int bit = 16 * (p & 1) + 2 * (2 * c + (p >> 1));
            if (to_packed) {
                const uint32_t q = (qs[32 * h + l] >> (2 * jq)) & 3u;
                words[t][G] |= q << bit;
            } else {
                const uint32_t q = (words[t][G] >> bit) & 3u;
                qs[32 * h + l] |= (uint8_t)(q << (2 * jq));
            }
        }
        if (to_packed)
            for (int t = 0; t < 4; ++t)
                for (int G = 0; G < 4; ++G) {
                    uint8_t *p = tb + 512 * hrow + 16 * (4 * g + t) + 4 * G;
                    for (int b = 0; b < 4; ++b) p[b] = (uint8_t)(words[t][G] >> (8 * b));
                }
        for (int sb = 0; sb < 16; ++sb) {
            uint8_t *p = tb + 1024 + 128 * hrow + 4 * (4 * g + (sb & 3)) + (sb >> 2);
            if (to_packed) *p = gguf[sb];
            else gguf[sb] = *p;
        }
        uint8_t *dd = tb + 1280 + 8 * g + 4 * hrow;
        for (int i = 0; i < 4; ++i) {
            if (to_packed) dd[i] = gguf[80 + i];
            else gguf[80 + i] = dd[i];
        }
        return;
    }
    if (qt == DS4G_Q4_K) {
        uint32_t words[4][8];  // [t][w]
        for (int t = 0; t < 4; ++t)
            for (int w = 0; w < 8; ++w) {
                uint8_t *p = tb + 1024 * hrow + 32 * (4 * g + t) + 4 * w;
                words[t][w] = to_packed ? 0u
                                        : (uint32_t)p[0] | ((uint32_t)p[1] << 8) |
                                              ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
            }
        uint8_t *qs = gguf + 16;
        if (!to_packed)
            for (int i = 0; i < 128; ++i) qs[i] = 0;
        for (int n = 0; n < 256; ++n) {
            const int c4 = n >> 6, r = n & 63;
            const int byte = 32 * c4 + (r & 31), shift = r < 32 ? 0 : 4;
            const int j = n >> 5, i = n & 31, t = j & 3, jj = j >> 2;
            const int c = i >> 2, p = i & 3;
            const int w = 4 * jj + (c >> 1);
            const int bit = 16 * (p & 1) + 4 * (2 * (c & 1) + (p >> 1));
            if (to_packed) {
                const uint32_t q = (qs[byte] >> shift) & 15u;
                words[t][w] |= q << bit;
            } else {
                const uint32_t q = (words[t][w] >> bit) & 15u;
                qs[byte] |= (uint8_t)(q << shift);
            }
        }
        if (to_packed)
            for (int t = 0; t < 4; ++t)
                for (int w = 0; w < 8; ++w) {
                    uint8_t *p = tb + 1024 * hrow + 32 * (4 * g + t) + 4 * w;
                    for (int b = 0; b < 4; ++b) p[b] = (uint8_t)(words[t][w] >> (8 * b));
                }
        uint8_t *sc = tb + 2048 + 12 * rr;
        for (int i = 0; i < 12; ++i) {
            if (to_packed) sc[i] = gguf[4 + i];
            else gguf[4 + i] = sc[i];
        }
        uint8_t *dd = tb + 2240 + 8 * g + 4 * hrow;
        for (int i = 0; i < 4; ++i) {
            if (to_packed) dd[i] = gguf[i];
            else gguf[i] = dd[i];
        }
    }
}

// One thread per (row, block).
__global__ void pack_kernel(int qt, int rows, int cols, const uint8_t *__restrict__ gguf,
                            uint8_t *__restrict__ packed) {
    const int nb = cols / 256;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)rows * nb) return;
    const int r = (int)(idx / nb), b = (int)(idx % nb);
    const int bb = gguf_block_bytes(qt), tbb = tile_block_bytes(qt);
    uint8_t blk[144];
    const uint8_t *src = gguf + ((size_t)r * nb + b) * bb;
    for (int i = 0; i < bb; ++i) blk[i] = src[i];
    uint8_t *tb = packed + ((size_t)(r >> 4) * nb + b) * tbb;
    map_block(qt, blk, tb, r & 15, true);
}

}  // namespace ds4g

using namespace ds4g;

static bool shape_ok(ds4g_qtype t, int rows, int cols) {
    return (t == DS4G_IQ2_XXS || t == DS4G_Q2_K || t == DS4G_Q4_K) && rows > 0 && cols > 0 &&
           rows % 16 == 0 && cols % 256 == 0;
}

extern "C" size_t ds4g_block_bytes(ds4g_qtype t) {
    return t == DS4G_BF16 ? 512 : (size_t)gguf_block_bytes(t);
}

extern "C" size_t ds4g_packed_size(ds4g_qtype t, int rows, int cols) {
    if (!shape_ok(t, rows, cols)) return 0;
    return (size_t)rows * (cols / 256) * gguf_block_bytes(t);
}

extern "C" ds4g_status ds4g_quantize_pack(ds4g_qtype t, int rows, int cols, const void *gguf_blocks,
                                          size_t in_bytes, void *packed, size_t out_bytes) {
    if (!gguf_blocks || !packed) return DS4G_EINVAL;
    if (t != DS4G_IQ2_XXS && t != DS4G_Q2_K && t != DS4G_Q4_K) return DS4G_EINVAL;
    if (!shape_ok(t, rows, cols)) return DS4G_EUNSUPPORTED;
    const size_t need = ds4g_packed_size(t, rows, cols);
    if (in_bytes < need || out_bytes < need) return DS4G_ENOSPACE;
    const int nb = cols / 256, bb = gguf_block_bytes(t), tbb = tile_block_bytes(t);
    uint8_t blk[144];
    for (int r = 0; r < rows; ++r)
        for (int b = 0; b < nb; ++b) {
            memcpy(blk, (const uint8_t *)gguf_blocks + ((size_t)r * nb + b) * bb, bb);
            uint8_t *tb = (uint8_t *)packed + ((size_t)(r >> 4) * nb + b) * tbb;
            map_block(t, blk, tb, r & 15, true);
        }
    return DS4G_OK;
}

extern "C" ds4g_status ds4g_unpack(ds4g_qtype t, int rows, int cols, const void *packed,
                                   size_t in_bytes, void *gguf_blocks, size_t out_bytes) {
    if (!gguf_blocks || !packed) return DS4G_EINVAL;
    if (t != DS4G_IQ2_XXS && t != DS4G_Q2_K && t != DS4G_Q4_K) return DS4G_EINVAL;
    if (!shape_ok(t, rows, cols)) return DS4G_EUNSUPPORTED;
    const size_t need = ds4g_packed_size(t, rows, cols);
    if (in_bytes < need || out_bytes < need) return DS4G_ENOSPACE;
    const int nb = cols / 256, bb = gguf_block_bytes(t), tbb = tile_block_bytes(t);
    uint8_t blk[144];
    for (int r = 0; r < rows; ++r)
        for (int b = 0; b < nb; ++b) {
            memset(blk, 0, sizeof blk);
            uint8_t *tb = (uint8_t *)packed + ((size_t)(r >> 4) * nb + b) * tbb;
            map_block(t, blk, tb, r & 15, false);
            memcpy((uint8_t *)gguf_blocks + ((size_t)r * nb + b) * bb, blk, bb);
        }
    return DS4G_OK;
}

extern "C" ds4g_status ds4g_quantize_pack_device(ds4g_qtype t, int rows, int cols,
                                                 const void *gguf_dev, void *packed_dev,
                                                 ds4g_stream_t s) {
    DS4G_TRACE();
    if (!gguf_dev || !packed_dev) return DS4G_EINVAL;
    if (t != DS4G_IQ2_XXS && t != DS4G_Q2_K && t != DS4G_Q4_K) return DS4G_EINVAL;
    if (!shape_ok(t, rows, cols)) return DS4G_EUNSUPPORTED;
    if (((uintptr_t)gguf_dev | (uintptr_t)packed_dev) & 15) return DS4G_EALIGN;
    const long long n = (long long)rows * (cols / 256);
    pack_kernel<<<(unsigned)((n + 127) / 128), 128, 0, (cudaStream_t)s>>>(
        t, rows, cols, (const uint8_t *)gguf_dev, (uint8_t *)packed_dev);
    return cudaGetLastError() == cudaSuccess ? DS4G_OK : DS4G_ECUDA;
}
