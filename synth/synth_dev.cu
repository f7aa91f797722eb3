// synth_dev.cu — CUDA twin of synth.gguf_matrix(): writes the same seeded
// GGUF-format block bytes straight into device memory (for multi-GB expert
// stacks).  Integer hashing plus the fp16 scale-field formula only; no part
// of the MoE computation lives here.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

static __host__ __device__ inline uint64_t splitmix64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// fp16 bits of 1e-3 + 3e-3 * u * 2^-24 for field number n (separate fp32
// roundings, then fp16 round-to-nearest-even).
static __device__ inline uint32_t scale_bits(uint64_t base_d, uint64_t n) {
    const uint32_t u = (uint32_t)(splitmix64(base_d + n) >> 40);
    float t = __fmul_rn(__uint2float_rn(u), 5.9604644775390625e-08f);
    t = __fmul_rn(3e-3f, t);
    const float d = __fadd_rn(1e-3f, t);
    return (uint32_t)__half_as_ushort(__float2half_rn(d));
}

// One thread per 8-byte word: the raw hash word, with every byte that belongs
// to an fp16 scale field replaced by that field's byte.
__global__ void fill_gguf(uint8_t *out, uint64_t nbytes, uint64_t base, uint64_t base_d, int bb,
                          int nf, int off0, int off1) {
    const uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const uint64_t pos0 = i * 8;
    if (pos0 >= nbytes) return;
    const uint64_t v = splitmix64(base + i);
    uint8_t bytes[8];
    for (int b = 0; b < 8; ++b) {
        const uint64_t pos = pos0 + b;
        uint8_t val = (uint8_t)(v >> (8 * b));
        const uint64_t blk = pos / (uint64_t)bb;
        const int off = (int)(pos % (uint64_t)bb);
        for (int f = 0; f < nf; ++f) {
            const int fo = f == 0 ? off0 : off1;
            if (off == fo || off == fo + 1) {
                const uint32_t bits = scale_bits(base_d, blk * nf + f);
                val = (uint8_t)(off == fo ? (bits & 0xffu) : (bits >> 8));
            }
        }
        bytes[b] = val;
    }
    for (int b = 0; b < 8 && pos0 + b < nbytes; ++b) out[pos0 + b] = bytes[b];
}

extern "C" int synth_fill_gguf(int qtype, int rows, int cols, uint64_t seed, uint64_t stream,
                               void *dev, void *cuda_stream) {
    int bb, nf, off0, off1 = 0;
    switch (qtype) {
    case 0: bb = 66; nf = 1; off0 = 0; break;              // IQ2_XXS
    case 1: bb = 84; nf = 2; off0 = 80; off1 = 82; break;  // Q2_K
    case 2: bb = 144; nf = 2; off0 = 0; off1 = 2; break;   // Q4_K
    default: return -1;
    }
    if (!dev || rows <= 0 || cols <= 0 || cols % 256) return -1;
    const uint64_t nblk = (uint64_t)rows * (cols / 256);
    const uint64_t nbytes = nblk * bb;
    const uint64_t base = seed ^ splitmix64(stream);
    const uint64_t base_d = seed ^ splitmix64(stream | (1ull << 63));
    const uint64_t nw = (nbytes + 7) / 8;
    fill_gguf<<<(unsigned)((nw + 255) / 256), 256, 0, (cudaStream_t)cuda_stream>>>(
        (uint8_t *)dev, nbytes, base, base_d, bb, nf, off0, off1);
    return cudaGetLastError() == cudaSuccess ? 0 : -2;
}
