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

// One thread per 8-byte word of the raw stream.
__global__ void fill_raw(uint8_t *out, uint64_t nbytes, uint64_t base) {
    const uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const uint64_t off = i * 8;
    if (off >= nbytes) return;
    const uint64_t v = splitmix64(base + i);
    if (off + 8 <= nbytes && (((uintptr_t)(out + off)) & 7) == 0) {
        *(uint64_t *)(out + off) = v;
    } else {
        for (int b = 0; b < 8 && off + b < nbytes; ++b) out[off + b] = (uint8_t)(v >> (8 * b));
    }
}

// One thread per fp16 scale field: fp16(1e-3 + 3e-3 * (h >> 40) * 2^-24).
__global__ void fill_fp16(uint8_t *out, uint64_t nblk, int bb, int nf, int off0, int off1,
                          uint64_t base_d) {
    const uint64_t n = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= nblk * (uint64_t)nf) return;
    const uint64_t blk = n / nf;
    const int fi = (int)(n % nf);
    const uint64_t u = splitmix64(base_d + n) >> 40;
    float t = __fmul_rn((float)u, 5.9604644775390625e-08f);  // * 2^-24, exact
    t = __fmul_rn(3e-3f, t);
    const float d = __fadd_rn(1e-3f, t);
    const uint16_t bits = __half_as_ushort(__float2half_rn(d));
    uint8_t *p = out + blk * bb + (fi == 0 ? off0 : off1);
    p[0] = (uint8_t)(bits & 0xff);
    p[1] = (uint8_t)(bits >> 8);
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
    cudaStream_t s = (cudaStream_t)cuda_stream;
    const uint64_t nblk = (uint64_t)rows * (cols / 256);
    const uint64_t nbytes = nblk * bb;
    const uint64_t base = seed ^ splitmix64(stream);
    const uint64_t base_d = seed ^ splitmix64(stream | (1ull << 63));
    const uint64_t nw = (nbytes + 7) / 8;
    fill_raw<<<(unsigned)((nw + 255) / 256), 256, 0, s>>>((uint8_t *)dev, nbytes, base);
    const uint64_t nfld = nblk * nf;
    fill_fp16<<<(unsigned)((nfld + 255) / 256), 256, 0, s>>>((uint8_t *)dev, nblk, bb, nf, off0,
                                                             off1, base_d);
    return cudaGetLastError() == cudaSuccess ? 0 : -2;
}
