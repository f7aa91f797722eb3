// ds4g_internal.cuh — shared definitions of the B300 routed-MoE library:
// fixed dimensions, the packed device layout of the quantised blocks, the
// workspace header, and small PTX wrappers (mma.sync, prmt, cache hints).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "../../include/ds4g.h"

namespace ds4g {

constexpr int kH = DS4G_N_EMBD;        // 4096
constexpr int kF = DS4G_N_FF_EXP;      // 2048
constexpr int kE = DS4G_N_EXPERT;      // 256
constexpr int kK = DS4G_N_EXPERT_USED; // 6
constexpr int kDecodeMaxT = 3;         // per-slot GEMV path handles T <= 3 (smem)
constexpr int kPrefillMinT = 64;       // from here on: bucketed tensor-core GEMM path

// ---------------------------------------------------------------------------
// Packed ("tile-block") layout.  A [rows][cols] matrix is cut into tiles of
// 16 rows x 256 cols; tile-block (rt, b) sits at byte (rt*cols/256 + b) * TB.
// Inside, a row rr (0..15) is addressed as g = rr & 7 (mma group id) and
// hrow = rr >> 3 (0: row g of the mma fragment, 1: row g+8).  Lane L = 4g + t
// of a warp owns the sub-blocks j == t (mod 4) of rows g and g+8, so every
// lane loads exactly the codes it feeds to the tensor core:
//   IQ2_XXS (TB 1056): [512*hrow + 16L + 8jj] = GGUF sub-block record 4jj+t
//            (4 grid-index bytes + 32-bit sign/scale word); d of rows g, g+8
//            at 1024 + 4g (+2 for g+8).
//   Q2_K   (TB 1344): [512*hrow + 16L + 4G] = 32-bit word of sub-block 4G+t:
//            2-bit quant of sub-block column i = 4c + p at bit
//            16*(p&1) + 2*(2c + (p>>1)); scale byte of sub-block 4G+t at
//            1024 + 128*hrow + 4L + G; (d, dmin) of row g, g+8 at
//            1280 + 8g (+4 for g+8).
//   Q4_K   (TB 2304): [1024*hrow + 32L + 4*(4jj + (c>>1))] = 32-bit word of
//            sub-block 4jj+t, column i = 4c + p at bit
//            16*(p&1) + 4*(2*(c&1) + (p>>1)); the 12 raw scale bytes of row rr
//            at 2048 + 12*rr; (d, dmin) of rows g, g+8 at 2240 + 8g (+4).
// Sizes equal the GGUF sizes (16 rows x 66/84/144 bytes per tile-block).
// ---------------------------------------------------------------------------
constexpr int kTB_IQ2 = 1056, kTB_Q2K = 1344, kTB_Q4K = 2304;

__host__ __device__ inline int gguf_block_bytes(int t) {
    return t == DS4G_IQ2_XXS ? 66 : t == DS4G_Q2_K ? 84 : t == DS4G_Q4_K ? 144 : 0;
}
__host__ __device__ inline int tile_block_bytes(int t) { return 16 * gguf_block_bytes(t); }

// ---------------------------------------------------------------------------
// Workspace header: first 256 bytes of every workspace.
//   [0]  uint32 status (ds4g_status of the first device-detected fault)
//   [1]  uint32 detail (e.g. the offending expert id)
// ---------------------------------------------------------------------------
constexpr size_t kWsHeader = 256;

// Counter area of the forward family's workspaces (ds4g_moe_forward, the
// fused layer kernel, the decode stack): after the status header come the
// fused kernel's coordination block and the per-slot decode kernels' tile
// counters, at the same offsets whatever T or path.  Every kernel leaves its
// counters at zero, and no path writes scratch below kWsScratch, so one
// zeroed workspace serves any sequence of calls and token counts.
constexpr size_t kWsD1Sync = kWsHeader;                      // decode1.cu coordination block
constexpr size_t kWsD1SyncBytes = 2048;
constexpr size_t kWsDecCnt = kWsD1Sync + kWsD1SyncBytes;     // decode.cu tile counters
constexpr size_t kWsDecCntBytes = 10752;
constexpr size_t kWsScratch = kWsDecCnt + kWsDecCntBytes;    // first byte of any path's scratch

__device__ inline void flag_status(uint32_t *ws_status, uint32_t code, uint32_t detail) {
    if (atomicCAS(ws_status, 0u, code) == 0u) ws_status[1] = detail;
}

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Tracing: every GPU entry point opens an NVTX range named after itself, so
// its launches group under that name in a profiler's timeline (Nsight
// Systems / Compute); with no tool attached a range costs a few nanoseconds.
struct TraceRange {
    explicit TraceRange(const char *name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange &) = delete;
    TraceRange &operator=(const TraceRange &) = delete;
};
#define DS4G_TRACE() ::ds4g::TraceRange ds4g_trace_range_(__func__)

// Decode path of the MoE block (decode.cu, 1 <= T <= 64): workspace bytes,
// and the launch of its kernels (phases: 1 gate/up, 2 down, 3 both).
// status_word: where its kernels record a fault (nullptr: the workspace's
// own header).  ready/epoch (streamed experts): the routed tasks of slot i
// wait until ready[i] == epoch (written by a copy stream after the slot's
// expert has landed); nullptr: no waiting.  q8: routed IQ2_XXS gate/up on
// int8 activations (ds4g_moe_forward_q8).
size_t decode_workspace(int T);
ds4g_status decode_forward(const float *hidden, int T, const ds4g_layer *L, const int32_t *ids, const float *w,
                           float *out, void *workspace, cudaStream_t st, int phases,
                           uint32_t *status_word = nullptr, const uint32_t *ready = nullptr, uint32_t epoch = 0,
                           int q8 = 0);

// ds4g_moe_forward's checks, then, for T <= kDecodeMaxT, the decode kernels
// with the ready flags above; DS4G_EUNSUPPORTED for larger T (api.cu).
ds4g_status forward_streamed_decode(const float *hidden, int T, const ds4g_layer *L, const int32_t *ids,
                                    const float *w, float *out, void *workspace, size_t ws_bytes, cudaStream_t st,
                                    const uint32_t *ready, uint32_t epoch);

// Batched decode path (batch.cu, 4 <= T < 64, IQ2_XXS gate/up and Q2_K
// down): the batch's slots grouped by expert, each selected expert read once
// per (up to 32-token) chunk.
size_t batch_workspace(int T);
ds4g_status batch_forward(const float *hidden, int T, const ds4g_layer *L, const int32_t *ids, const float *w,
                          float *out, void *workspace, cudaStream_t st);

// TMA tensor maps over a row-major [rows][cols] bf16 matrix, 128-byte
// swizzle (tmap.cu).  tmap_bf16_2d: box of 64 columns x box_rows rows.
// tmap_bf16_rowtile: box of tile_rows rows x (64 * tile_chunks) columns,
// landing in shared memory as [tile_chunks][tile_rows][64] (one 128-byte line
// per row of a 64-column chunk, so the swizzle rotates 16-byte units by row).
// False if the encoder is unavailable or refuses the arguments.
bool tmap_bf16_2d(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows);
bool tmap_bf16_rowtile(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t tile_rows,
                       uint32_t tile_chunks);

// An expert id is usable if it is in range and its packed matrices are
// non-NULL and 16-byte aligned (a misaligned vector load would fault).
__device__ __forceinline__ bool expert_ok(int e, const void *const *a, const void *const *b,
                                          const void *const *c) {
    if ((unsigned)e >= (unsigned)kE) return false;
    const uintptr_t pa = (uintptr_t)a[e], pb = b ? (uintptr_t)b[e] : 16, pc = c ? (uintptr_t)c[e] : 16;
    return pa && pb && pc && !((pa | pb | pc) & 15);
}

// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// D = A * B + C, m16n8k16, A/B f16, accumulate f32.
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Same with bf16 operands.
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Streaming loads of weights (read once): do not allocate in L1.
__device__ __forceinline__ uint4 ldg_stream128(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ uint2 ldg_stream64(const void *p) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(r.x), "=r"(r.y)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ uint32_t ldg_stream32(const void *p) {
    uint32_t r;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

// 0.5 + (float)n for a 4-bit n without an int->float conversion:
// 2^23 + n has n in the low mantissa bits.
__device__ __forceinline__ float half_plus(uint32_t n) {
    return __uint_as_float(0x4B000000u | n) - 8388607.5f;
}
__device__ __forceinline__ float small_u2f(uint32_t n) {  // exact for n < 2^23
    return __uint_as_float(0x4B000000u | n) - 8388608.0f;
}

// fp32 -> (hi, lo) pair with hi = rn(x), lo = rn(x - hi).
__device__ __forceinline__ void split_f16(float x, __half &hi, __half &lo) {
    hi = __float2half_rn(x);
    lo = __float2half_rn(x - __half2float(hi));
}
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16 &hi, __nv_bfloat16 &lo) {
    hi = __float2bfloat16_rn(x);
    lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

__device__ __forceinline__ float silu_f(float v) { return v / (1.0f + expf(-v)); }

// Exponent e >= 0 such that every |h| <= m of a group, scaled by 2^-e, is
// below 2^15 (then its fp16 hi/lo pair is exact to ~2^-22 of the group's
// largest value); e = 0 when m < 2^15.  The routed h of the decode paths is
// stored as 2^-e * h per 16 entries, with 2^e beside it.
__device__ __forceinline__ int h_group_exp(float m) {
    const int E = (int)((__float_as_uint(m) >> 23) & 255u) - 126;   // m < 2^E for normal m
    return E > 15 ? E - 15 : 0;
}
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

}  // namespace ds4g
