// decode.cu — the MoE block for small T (decode; chenxutan ds4 article §3.2:
// router result -> only the routed experts' weights are read -> shared expert
// -> merge).  Two persistent kernels, one CTA of 16 warps per SM:
//
//  gate/up: warp tasks are (slot, 16-row tile, 512-col split) of a routed
//    expert (IQ2_XXS or Q4_K) or (16-row tile, 128-col split) of the bf16
//    shared expert.  Each task streams its weights straight into registers
//    with 128-bit loads, decodes the codes in registers into mma.sync A
//    fragments and multiplies by the token's activation.  The last task to
//    finish a tile (atomic ticket) sums the split partials in a fixed order,
//    applies SwiGLU and writes h.
//  down: tasks are (token, 16-row tile, 256-col block) over that token's six
//    routed experts (Q2_K or Q4_K; routing weight folded in) or (16-row tile,
//    256-col block) of the bf16 shared expert; the last task of a tile writes
//    out = shared + sum_k w_k y_k for its 16 rows.  No atomics touch values.
//
// Exact dequantisation on the tensor cores: an IQ2 grid value g (<= 43), a
// Q2_K quant q (<= 3) or a Q4_K quant (<= 15) is placed in the mantissa of an
// fp16 subnormal (value g * 2^-24, sign bit from the sign table) with one
// prmt / and, so the mma sums code * x without rounding the codes; the block
// and sub-block scales (and Q2_K/Q4_K mins via per-sub-block sums of the
// activation) are applied to the fp32 results.  The activation enters as an
// fp16 hi + lo pair (about 22 significant bits).  Because each routed slot has
// exactly one token, the 8 mma columns carry (hi, lo) for the sub-blocks of
// the 4 lanes of a quad ("block-diagonal B"), so each lane gets the sums of
// its own sub-blocks and applies its own scales.
#include "ds4g_internal.cuh"

namespace ds4g {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kTilesGU = kF / 16;    // 128 row tiles of gate/up
constexpr int kTilesDN = kH / 16;    // 256 row tiles of down
constexpr int kSplitR = 8;           // routed gate/up: 8 splits of 512 cols
constexpr int kSplitS = 32;          // shared gate/up: 32 splits of 128 cols
constexpr int kBlkDN = kF / 256;     // 8 blocks of 256 cols in down

struct DecodeArgs {
    const float *x;
    int T;
    const int32_t *ids;
    const float *w;
    int gu_type, dn_type;
    const uint8_t *const *gate;
    const uint8_t *const *up;
    const uint8_t *const *down;
    const __nv_bfloat16 *sh_gate, *sh_up, *sh_down;
    const uint64_t *grid;
    float *out;
    uint32_t *status;
    uint32_t *cnt_gu;     // [(6T+1)][128]
    uint32_t *cnt_dn;     // [256]
    float *part_r;        // [6T][128][kSplitR][2][16]
    float *part_s;        // [128][kSplitS][2][T][16]
    __half *hq;           // [6T][2][2048]  routed h as fp16 (hi, lo)
    float *xs16;          // [6T][8][4][4]  sums of h over 16 consecutive entries
    float *hsc16;         // [6T][8][4][4]  power-of-two scale of each 16 entries of hq (layout of xs16)
    __nv_bfloat16 *hs;    // [T][2][2048]   shared h as bf16 (hi, lo)
    float *part_dr;       // [T][256][8][16]
    float *part_ds;       // [256][8][T][16]
    const uint32_t *ready; // streamed experts: ready[slot] == epoch once the slot's expert has landed (or NULL)
    uint32_t epoch;
    int q8;               // routed IQ2_XXS gate/up on int8 activations (dp4a)
};

// Streamed experts (ds4g_moe_forward_streamed): a copy stream writes
// ready[slot] = epoch after the slot's expert (gate, up, down) has been copied
// into its cache slot, while this kernel already runs the shared expert.
// Lane 0 waits for it (bounded: ~1 s, then DS4G_ETIMEOUT) before the warp
// reads the expert.  The flag follows the expert's copies on that stream, and
// the expert is read through L2 (no L1 allocation), so the data is there.
__device__ __forceinline__ void wait_expert(const DecodeArgs &a, int slot) {
    if (!a.ready) return;
    if ((threadIdx.x & 31) == 0) {
        const long long t0 = clock64();
        while (true) {
            uint32_t v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a.ready + slot) : "memory");
            if (v == a.epoch) break;
            if (clock64() - t0 > (2ll << 30)) {
                flag_status(a.status, DS4G_ETIMEOUT, 0x5700u + (uint32_t)slot);
                break;
            }
            __nanosleep(256);
        }
    }
    __syncwarp();
}

// ------------------------------------------------------------- task mixing
// Interleave the two task kinds evenly (Bresenham) so every SM sees the same
// mix of lookup-heavy routed work and bandwidth-heavy bf16 work.
__device__ __forceinline__ bool task_kind(long long tau, long long NR, long long NS, long long &idx) {
    const long long N = NR + NS;
    const long long sb = tau * NS / N, sa = (tau + 1) * NS / N;
    if (sa > sb) {
        idx = sb;
        return true;  // shared
    }
    idx = tau - sb;
    return false;
}

// ------------------------------------------------------- ticket for a tile
// Every lane that wrote partials fences; lane 0 takes a ticket; returns true
// in all lanes of the warp that took the last ticket.
__device__ __forceinline__ bool last_arrival(uint32_t *cnt, uint32_t target) {
    __threadfence();
    __syncwarp();
    uint32_t ticket = 0;
    if ((threadIdx.x & 31) == 0) ticket = atomicAdd(cnt, 1u);
    ticket = __shfl_sync(0xffffffffu, ticket, 0);
    const bool last = ticket == target - 1;
    if (last) {
        __threadfence();
        if ((threadIdx.x & 31) == 0) *cnt = 0u;  // ready for the next call
    }
    return last;
}

// ===================================================================== gate/up
struct GUSmem {
    uint2 *gtab;  // [256][16] grid rows, 16 replicas (lane & 15) -> conflict-free
    uint2 *stab;  // [128][16] sign bytes (0x80 / 0x00) of each 7-bit sign index
    __half *xq;   // [T][2][4096] activation fp16 (hi, lo)
    __nv_bfloat16 *xb;  // [T][2][4096] activation bf16 (hi, lo)
    // q8 only:
    uint4 *stab8;  // [128][16] per sign index: 0xFF / 0x00 masks (bytes 0-3, 4-7), then 0x01 / 0x00
    int8_t *x8;    // [T][4096] activation as int8 (blocks of 256)
    float *dx;     // [T][16] the blocks' scales
};

// Reduction of one (slot, tile) of routed gate/up: 8 split partials in fixed
// order -> h = silu(g) * u; the 16 values, scaled by a power of two 2^-e
// shared by the tile (so that any finite h fits the fp16 range), as fp16
// hi/lo; 2^e; and the 16-row sum of the unscaled h.
__device__ __forceinline__ void gu_routed_finish(const DecodeArgs &a, int slot, int tile) {
    const int lane = threadIdx.x & 31;
    float h = 0.f;
    if (lane < 16) {
        const float *base = a.part_r + ((size_t)slot * kTilesGU + tile) * kSplitR * 32;
        float gs = 0.f, us = 0.f;
#pragma unroll
        for (int s = 0; s < kSplitR; ++s) {
            gs += __ldcg(base + s * 32 + lane);
            us += __ldcg(base + s * 32 + 16 + lane);
        }
        h = silu_f(gs) * us;
        if (!(fabsf(h) <= 3.4028235e38f)) flag_status(a.status, DS4G_EDEVICE, 0xF16u);   // inf or NaN
    }
    float m = fabsf(h);
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const int e = h_group_exp(m);
    const int b = tile >> 4, j = tile & 15;
    if (lane < 16) {
        __half hi, lo;
        split_f16(h * pow2f(-e), hi, lo);
        a.hq[((size_t)slot * 2 + 0) * kF + tile * 16 + lane] = hi;
        a.hq[((size_t)slot * 2 + 1) * kF + tile * 16 + lane] = lo;
    }
    // sum of h over the 16 rows = one 16-col sub-block of the down matrix
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) h += __shfl_xor_sync(0xffffffffu, h, off);
    if (lane == 0) {
        a.xs16[(size_t)slot * 128 + (b * 4 + (j & 3)) * 4 + (j >> 2)] = h;
        a.hsc16[(size_t)slot * 128 + (b * 4 + (j & 3)) * 4 + (j >> 2)] = pow2f(e);
    }
}

__device__ __forceinline__ void gu_write_partial(const DecodeArgs &a, int slot, int tile, int split,
                                                 float (&acc)[2][2]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            acc[m][h] += __shfl_xor_sync(0xffffffffu, acc[m][h], 1);
            acc[m][h] += __shfl_xor_sync(0xffffffffu, acc[m][h], 2);
        }
    float *pp = a.part_r + (((size_t)slot * kTilesGU + tile) * kSplitR + split) * 32;
    if (t == 0) {
        pp[g] = acc[0][0];
        pp[g + 8] = acc[0][1];
        pp[16 + g] = acc[1][0];
        pp[16 + g + 8] = acc[1][1];
    }
    if (last_arrival(a.cnt_gu + (size_t)slot * kTilesGU + tile, kSplitR)) gu_routed_finish(a, slot, tile);
}

__device__ __forceinline__ void gu_routed_iq2(const DecodeArgs &a, const GUSmem &sm, long long r) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3, p = lane & 15;
    const int slot = (int)(r / (kTilesGU * kSplitR));
    const int rem = (int)(r % (kTilesGU * kSplitR));
    const int tile = rem / kSplitR, split = rem % kSplitR;
    const int e = a.ids[slot];
    wait_expert(a, slot);
    float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};  // [matrix][row g / g+8]
    if (expert_ok(e, (const void *const *)a.gate, (const void *const *)a.up, nullptr)) {
        const uint8_t *mat[2] = {a.gate[e], a.up[e]};
        uint4 qa[2][2], qb[2][2];
        uint32_t dd[2][2];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2) {
                const uint8_t *tb = mat[m] + ((size_t)tile * 16 + 2 * split + s2) * kTB_IQ2;
                qa[m][s2] = ldg_stream128(tb + 16 * lane);
                qb[m][s2] = ldg_stream128(tb + 512 + 16 * lane);
                dd[m][s2] = ldg_stream32(tb + 1024 + 4 * g);
            }
        const int tok = slot / kK;
        const bool active = (g >> 1) == t;
        const __half *xrow = sm.xq + ((size_t)tok * 2 + (g & 1)) * kH;
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
            const int b = 2 * split + s2;
            uint32_t B[2][16];
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const uint4 *src = reinterpret_cast<const uint4 *>(xrow + 256 * b + 32 * (4 * jj + t));
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 v = active ? src[q] : make_uint4(0, 0, 0, 0);
                    B[jj][4 * q + 0] = v.x;
                    B[jj][4 * q + 1] = v.y;
                    B[jj][4 * q + 2] = v.z;
                    B[jj][4 * q + 3] = v.w;
                }
            }
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                // d * 0.25 * 2^24 (the codes enter the mma as code * 2^-24)
                const float d4g = __half2float(__ushort_as_half((unsigned short)(dd[m][s2] & 0xffffu))) * 4194304.0f;
                const float d4h = __half2float(__ushort_as_half((unsigned short)(dd[m][s2] >> 16))) * 4194304.0f;
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const uint32_t ia = jj ? qa[m][s2].z : qa[m][s2].x, va = jj ? qa[m][s2].w : qa[m][s2].y;
                    const uint32_t ib = jj ? qb[m][s2].z : qb[m][s2].x, vb = jj ? qb[m][s2].w : qb[m][s2].y;
                    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int l = 0; l < 4; ++l) {
                        const uint2 ga = sm.gtab[((ia >> (8 * l)) & 255u) * 16 + p];
                        const uint2 sa = sm.stab[((va >> (7 * l)) & 127u) * 16 + p];
                        const uint2 gb = sm.gtab[((ib >> (8 * l)) & 255u) * 16 + p];
                        const uint2 sbv = sm.stab[((vb >> (7 * l)) & 127u) * 16 + p];
#pragma unroll
                        for (int mm = 0; mm < 2; ++mm) {
                            const uint32_t gA = mm ? ga.y : ga.x, sA = mm ? sa.y : sa.x;
                            const uint32_t gB = mm ? gb.y : gb.x, sB = mm ? sbv.y : sbv.x;
                            mma_f16(c, prmt(gA, sA, 0x5140), prmt(gB, sB, 0x5140), prmt(gA, sA, 0x7362),
                                    prmt(gB, sB, 0x7362), B[jj][2 * (2 * l + mm)], B[jj][2 * (2 * l + mm) + 1]);
                        }
                    }
                    acc[m][0] = fmaf(d4g * half_plus(va >> 28), c[0] + c[1], acc[m][0]);
                    acc[m][1] = fmaf(d4h * half_plus(vb >> 28), c[2] + c[3], acc[m][1]);
                }
            }
        }
    } else if (lane == 0) {
        flag_status(a.status, DS4G_EDEVICE, (uint32_t)e);
    }
    gu_write_partial(a, slot, tile, split, acc);
}

// IQ2_XXS gate/up on int8 activations (the int8 path: chenxutan ds4 article
// §2.4, dot_iq2_pair_16: int8 grid values against int8 activations).  x is
// held as q8 (blocks of 256: q = x / d to nearest, ties to even, d =
// max|x| / 127).  Lane (g, t) owns sub-blocks 4jj + t of rows g and g + 8 (the
// packed layout's ownership) and forms each sub-block's exact integer sum
// S = sum (sign * grid value) * q with dp4a: a negative byte is taken as
// (g ^ 0xFF) = -g - 1 and the +1 is added back by a dp4a of the 0x01 mask.
// Then acc += (d (0.5 + ls) 0.25) * d_x * S in fp32.
__device__ __forceinline__ void gu_routed_iq2_q8(const DecodeArgs &a, const GUSmem &sm, long long r) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3, p = lane & 15;
    const int slot = (int)(r / (kTilesGU * kSplitR));
    const int rem = (int)(r % (kTilesGU * kSplitR));
    const int tile = rem / kSplitR, split = rem % kSplitR;
    const int e = a.ids[slot];
    wait_expert(a, slot);
    float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    if (expert_ok(e, (const void *const *)a.gate, (const void *const *)a.up, nullptr)) {
        const uint8_t *mat[2] = {a.gate[e], a.up[e]};
        uint4 qa[2][2], qb[2][2];
        uint32_t dd[2][2];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2) {
                const uint8_t *tb = mat[m] + ((size_t)tile * 16 + 2 * split + s2) * kTB_IQ2;
                qa[m][s2] = ldg_stream128(tb + 16 * lane);
                qb[m][s2] = ldg_stream128(tb + 512 + 16 * lane);
                dd[m][s2] = ldg_stream32(tb + 1024 + 4 * g);
            }
        const int tok = slot / kK;
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
            const int b = 2 * split + s2;
            const float dxb = sm.dx[tok * 16 + b];
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int j = 4 * jj + t;
                const uint4 *xs = reinterpret_cast<const uint4 *>(sm.x8 + (size_t)tok * kH + 256 * b + 32 * j);
                const uint4 x0 = xs[0], x1 = xs[1];
                const int xw[8] = {(int)x0.x, (int)x0.y, (int)x0.z, (int)x0.w,
                                   (int)x1.x, (int)x1.y, (int)x1.z, (int)x1.w};
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    const uint32_t ia = jj ? qa[m][s2].z : qa[m][s2].x, va = jj ? qa[m][s2].w : qa[m][s2].y;
                    const uint32_t ib = jj ? qb[m][s2].z : qb[m][s2].x, vb = jj ? qb[m][s2].w : qb[m][s2].y;
                    int Sa = 0, Sb = 0;
#pragma unroll
                    for (int l = 0; l < 4; ++l) {
                        const uint2 ga = sm.gtab[((ia >> (8 * l)) & 255u) * 16 + p];
                        const uint4 sa = sm.stab8[((va >> (7 * l)) & 127u) * 16 + p];
                        const uint2 gb = sm.gtab[((ib >> (8 * l)) & 255u) * 16 + p];
                        const uint4 sb = sm.stab8[((vb >> (7 * l)) & 127u) * 16 + p];
                        Sa = __dp4a((int)(ga.x ^ sa.x), xw[2 * l], Sa);
                        Sa = __dp4a((int)(ga.y ^ sa.y), xw[2 * l + 1], Sa);
                        Sa = __dp4a((int)sa.z, xw[2 * l], Sa);
                        Sa = __dp4a((int)sa.w, xw[2 * l + 1], Sa);
                        Sb = __dp4a((int)(gb.x ^ sb.x), xw[2 * l], Sb);
                        Sb = __dp4a((int)(gb.y ^ sb.y), xw[2 * l + 1], Sb);
                        Sb = __dp4a((int)sb.z, xw[2 * l], Sb);
                        Sb = __dp4a((int)sb.w, xw[2 * l + 1], Sb);
                    }
                    const float dga = __half2float(__ushort_as_half((unsigned short)(dd[m][s2] & 0xffffu)));
                    const float dgb = __half2float(__ushort_as_half((unsigned short)(dd[m][s2] >> 16)));
                    const float dba = __fmul_rn(__fmul_rn(dga, half_plus(va >> 28)), 0.25f);
                    const float dbb = __fmul_rn(__fmul_rn(dgb, half_plus(vb >> 28)), 0.25f);
                    acc[m][0] = fmaf(dba * dxb, (float)Sa, acc[m][0]);
                    acc[m][1] = fmaf(dbb * dxb, (float)Sb, acc[m][1]);
                }
            }
        }
    } else if (lane == 0) {
        flag_status(a.status, DS4G_EDEVICE, (uint32_t)e);
    }
    gu_write_partial(a, slot, tile, split, acc);
}

// Q4_K gate/up (q4 layers): lane sub-blocks 4jj+t of 32 cols, 8 chunks each.
__device__ __forceinline__ void gu_routed_q4k(const DecodeArgs &a, const GUSmem &sm, long long r) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int slot = (int)(r / (kTilesGU * kSplitR));
    const int rem = (int)(r % (kTilesGU * kSplitR));
    const int tile = rem / kSplitR, split = rem % kSplitR;
    const int e = a.ids[slot];
    wait_expert(a, slot);
    float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    if (expert_ok(e, (const void *const *)a.gate, (const void *const *)a.up, nullptr)) {
        const uint8_t *mat[2] = {a.gate[e], a.up[e]};
        const int tok = slot / kK;
        const bool active = (g >> 1) == t;
        const __half *xrow = sm.xq + ((size_t)tok * 2 + (g & 1)) * kH;
#pragma unroll 1
        for (int s2 = 0; s2 < 2; ++s2) {
            const int b = 2 * split + s2;
            uint4 q[2][2][2];  // [m][hrow][jj]
            uint32_t scw[2][2][3];
            uint2 dd[2];
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const uint8_t *tb = mat[m] + ((size_t)tile * 16 + b) * kTB_Q4K;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    q[m][h][0] = ldg_stream128(tb + 1024 * h + 32 * lane);
                    q[m][h][1] = ldg_stream128(tb + 1024 * h + 32 * lane + 16);
#pragma unroll
                    for (int i = 0; i < 3; ++i)
                        scw[m][h][i] = ldg_stream32(tb + 2048 + 12 * (g + 8 * h) + 4 * i);
                }
                dd[m] = ldg_stream64(tb + 2240 + 8 * g);
            }
            uint32_t B[2][16];
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const uint4 *src = reinterpret_cast<const uint4 *>(xrow + 256 * b + 32 * (4 * jj + t));
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    const uint4 v = active ? src[qq] : make_uint4(0, 0, 0, 0);
                    B[jj][4 * qq + 0] = v.x;
                    B[jj][4 * qq + 1] = v.y;
                    B[jj][4 * qq + 2] = v.z;
                    B[jj][4 * qq + 3] = v.w;
                }
            }
            // sums of the activation (hi + lo) over the lane's sub-blocks, for
            // the mins; computed by the "hi" lane 9t of each quad, shared
            float xsum[2] = {0.f, 0.f};
            if (active && (g & 1) == 0) {
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    float s = 0.f;
                    const int c0 = 256 * b + 32 * (4 * jj + t);
                    const __half *xh = sm.xq + ((size_t)tok * 2) * kH + c0;
                    const __half *xl = xh + kH;
                    for (int i = 0; i < 32; ++i) s += __half2float(xh[i]) + __half2float(xl[i]);
                    xsum[jj] = s;
                }
            }
            const float xs0 = __shfl_sync(0xffffffffu, xsum[0], 9 * t);
            const float xs1 = __shfl_sync(0xffffffffu, xsum[1], 9 * t);
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const float dgv[2] = {__half2float(__ushort_as_half((unsigned short)(dd[m].x & 0xffff))) * 16777216.0f,
                                      __half2float(__ushort_as_half((unsigned short)(dd[m].y & 0xffff))) * 16777216.0f};
                const float dmv[2] = {__half2float(__ushort_as_half((unsigned short)(dd[m].x >> 16))),
                                      __half2float(__ushort_as_half((unsigned short)(dd[m].y >> 16)))};
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int j = 4 * jj + t;
                    float c[4] = {0.f, 0.f, 0.f, 0.f};
                    const uint32_t wa[4] = {q[m][0][jj].x, q[m][0][jj].y, q[m][0][jj].z, q[m][0][jj].w};
                    const uint32_t wb[4] = {q[m][1][jj].x, q[m][1][jj].y, q[m][1][jj].z, q[m][1][jj].w};
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        const uint32_t Wa = wa[cc >> 1], Wb = wb[cc >> 1];
                        const int s0 = 8 * (cc & 1);
                        mma_f16(c, (Wa >> s0) & 0x000F000Fu, (Wb >> s0) & 0x000F000Fu,
                                (Wa >> (s0 + 4)) & 0x000F000Fu, (Wb >> (s0 + 4)) & 0x000F000Fu,
                                B[jj][2 * cc], B[jj][2 * cc + 1]);
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        // sub-block j needs scale bytes s[j], s[j+4], s[j+8]:
                        // byte (j & 3) of the row's three scale words
                        const uint32_t s0 = (scw[m][h][0] >> (8 * (j & 3))) & 0xffu;
                        const uint32_t s1 = (scw[m][h][1] >> (8 * (j & 3))) & 0xffu;
                        const uint32_t s2b = (scw[m][h][2] >> (8 * (j & 3))) & 0xffu;
                        uint32_t sc, mn;
                        if (j < 4) {
                            sc = s0 & 63u;
                            mn = s1 & 63u;
                        } else {
                            sc = (s2b & 15u) | ((s0 >> 6) << 4);
                            mn = (s2b >> 4) | ((s1 >> 6) << 4);
                        }
                        const float dot = h ? (c[2] + c[3]) : (c[0] + c[1]);
                        acc[m][h] += dgv[h] * small_u2f(sc) * dot - dmv[h] * small_u2f(mn) * (jj ? xs1 : xs0);
                    }
                }
            }
        }
    } else if (lane == 0) {
        flag_status(a.status, DS4G_EDEVICE, (uint32_t)e);
    }
    gu_write_partial(a, slot, tile, split, acc);
}

// bf16 shared expert gate/up task: 16 rows x 128 cols of Sg and Su, all tokens.
__device__ __forceinline__ void gu_shared(const DecodeArgs &a, const GUSmem &sm, long long s) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int tile = (int)(s / kSplitS), split = (int)(s % kSplitS);
    const int col0 = 128 * split;
    const __nv_bfloat16 *mats[2] = {a.sh_gate, a.sh_up};
    uint2 A[2][8][2];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                A[m][ch][h] = ldg_stream64(mats[m] + (size_t)(tile * 16 + g + 8 * h) * kH + col0 + 16 * ch + 4 * t);
    const int tok = g >> 1;
    const bool has = tok < a.T;
    const __nv_bfloat16 *xrow = sm.xb + ((size_t)(has ? tok : 0) * 2 + (g & 1)) * kH + col0 + 4 * t;
    float c[2][4] = {};
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        const uint2 bv = has ? *reinterpret_cast<const uint2 *>(xrow + 16 * ch) : make_uint2(0, 0);
#pragma unroll
        for (int m = 0; m < 2; ++m)
            mma_bf16(c[m], A[m][ch][0].x, A[m][ch][1].x, A[m][ch][0].y, A[m][ch][1].y, bv.x, bv.y);
    }
    float *pp = a.part_s + ((size_t)tile * kSplitS + split) * 2 * a.T * 16;
    if (t < a.T) {
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            pp[(m * a.T + t) * 16 + g] = c[m][0] + c[m][1];
            pp[(m * a.T + t) * 16 + g + 8] = c[m][2] + c[m][3];
        }
    }
    if (!last_arrival(a.cnt_gu + (size_t)kK * a.T * kTilesGU + tile, kSplitS)) return;
    for (int i = lane; i < 16 * a.T; i += 32) {
        const int rr = i & 15, tk = i >> 4;
        const float *base = a.part_s + (size_t)tile * kSplitS * 2 * a.T * 16;
        float gs = 0.f, us = 0.f;
        for (int sp = 0; sp < kSplitS; ++sp) {
            gs += __ldcg(base + ((size_t)sp * 2 * a.T + tk) * 16 + rr);
            us += __ldcg(base + ((size_t)sp * 2 * a.T + a.T + tk) * 16 + rr);
        }
        const float h = silu_f(gs) * us;
        __nv_bfloat16 hi, lo;
        split_bf16(h, hi, lo);
        a.hs[((size_t)tk * 2 + 0) * kF + tile * 16 + rr] = hi;
        a.hs[((size_t)tk * 2 + 1) * kF + tile * 16 + rr] = lo;
    }
}

__global__ void __launch_bounds__(kThreads, 1) gateup_decode_kernel(DecodeArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    GUSmem sm;
    sm.gtab = reinterpret_cast<uint2 *>(smem_raw);
    sm.stab = sm.gtab + 256 * 16;
    sm.xq = reinterpret_cast<__half *>(sm.stab + 128 * 16);
    sm.xb = reinterpret_cast<__nv_bfloat16 *>(sm.xq + (size_t)a.T * 2 * kH);
    sm.stab8 = reinterpret_cast<uint4 *>(sm.xb + (size_t)a.T * 2 * kH);
    sm.x8 = reinterpret_cast<int8_t *>(sm.stab8 + 128 * 16);
    sm.dx = reinterpret_cast<float *>(sm.x8 + (size_t)a.T * kH);
    const int tid = threadIdx.x;
    if (a.gu_type == DS4G_IQ2_XXS) {
        for (int i = tid; i < 256 * 16; i += kThreads) {
            const uint64_t row = a.grid[i >> 4];
            sm.gtab[i] = make_uint2((uint32_t)row, (uint32_t)(row >> 32));
        }
        for (int i = tid; i < 128 * 16; i += kThreads) {
            const uint32_t s7 = (uint32_t)(i >> 4);
            const uint32_t sg = s7 | ((uint32_t)(__popc(s7) & 1) << 7);
            uint32_t lo = 0, hi = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                lo |= ((sg >> j) & 1u) << (8 * j + 7);
                hi |= ((sg >> (j + 4)) & 1u) << (8 * j + 7);
            }
            sm.stab[i] = make_uint2(lo, hi);
            if (a.q8) {
                uint32_t mlo = 0, mhi = 0, olo = 0, ohi = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    mlo |= ((sg >> j) & 1u) * (0xFFu << (8 * j));
                    mhi |= ((sg >> (j + 4)) & 1u) * (0xFFu << (8 * j));
                    olo |= ((sg >> j) & 1u) << (8 * j);
                    ohi |= ((sg >> (j + 4)) & 1u) << (8 * j);
                }
                sm.stab8[i] = make_uint4(mlo, mhi, olo, ohi);
            }
        }
    }
    if (a.q8) {
        // q8 activations: per token and 256-column block, d = max|x| / 127,
        // q = x / d to nearest (ties to even), clamped to +-127; one warp per block
        const int wid = tid >> 5, lane = tid & 31;
        for (int blk = wid; blk < a.T * 16; blk += kWarps) {
            const int tk = blk >> 4, b = blk & 15;
            const float *xr = a.x + (size_t)tk * kH + 256 * b;
            float v[8], amax = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                v[i] = xr[lane + 32 * i];
                amax = fmaxf(amax, fabsf(v[i]));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const float db = __fdiv_rn(amax, 127.0f);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                int q = 0;
                if (db > 0.f) q = max(-127, min(127, __float2int_rn(__fdiv_rn(v[i], db))));
                sm.x8[(size_t)tk * kH + 256 * b + lane + 32 * i] = (int8_t)q;
            }
            if (lane == 0) sm.dx[tk * 16 + b] = db;
        }
    }
    for (int i = tid; i < a.T * kH; i += kThreads) {
        const float v = a.x[i];
        if (!(fabsf(v) < 65504.f)) flag_status(a.status, DS4G_EDEVICE, 0xF16u);
        const int tk = i / kH, c = i % kH;
        __half hi, lo;
        split_f16(v, hi, lo);
        sm.xq[((size_t)tk * 2) * kH + c] = hi;
        sm.xq[((size_t)tk * 2 + 1) * kH + c] = lo;
        __nv_bfloat16 bh, bl;
        split_bf16(v, bh, bl);
        sm.xb[((size_t)tk * 2) * kH + c] = bh;
        sm.xb[((size_t)tk * 2 + 1) * kH + c] = bl;
    }
    __syncthreads();
    const long long NR = (long long)kK * a.T * kTilesGU * kSplitR;
    const long long NS = (long long)kTilesGU * kSplitS;
    const long long W = (long long)gridDim.x * kWarps;
    for (long long tau = blockIdx.x * kWarps + (tid >> 5); tau < NR + NS; tau += W) {
        long long idx;
        bool sh;
        if (a.ready) {
            // streamed experts: the shared expert's tasks first, while the
            // routed experts are still being copied
            sh = tau < NS;
            idx = sh ? tau : tau - NS;
        } else {
            sh = task_kind(tau, NR, NS, idx);
        }
        if (sh) gu_shared(a, sm, idx);
        else if (a.gu_type == DS4G_IQ2_XXS && a.q8) gu_routed_iq2_q8(a, sm, idx);
        else if (a.gu_type == DS4G_IQ2_XXS) gu_routed_iq2(a, sm, idx);
        else gu_routed_q4k(a, sm, idx);
    }
}

// ======================================================================= down
struct DNSmem {
    __half *hq;          // [6T][2][2048]
    float *xs;           // [6T][128]
    float *hsc;          // [6T][128] scale of each 16 entries of hq
    __nv_bfloat16 *hs;   // [T][2][2048]
};

__device__ __forceinline__ void dn_finish(const DecodeArgs &a, int tile) {
    const int lane = threadIdx.x & 31;
    for (int i = lane; i < 16 * a.T; i += 32) {
        const int rr = i & 15, tk = i >> 4;
        float v = 0.f;
        for (int b = 0; b < kBlkDN; ++b) v += __ldcg(a.part_ds + (((size_t)tile * kBlkDN + b) * a.T + tk) * 16 + rr);
        for (int b = 0; b < kBlkDN; ++b) v += __ldcg(a.part_dr + (((size_t)tk * kTilesDN + tile) * kBlkDN + b) * 16 + rr);
        a.out[(size_t)tk * kH + tile * 16 + rr] = v;
    }
}

__device__ __forceinline__ void dn_write_partial(const DecodeArgs &a, int tok, int tile, int b, float (&racc)[2]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        racc[h] += __shfl_xor_sync(0xffffffffu, racc[h], 1);
        racc[h] += __shfl_xor_sync(0xffffffffu, racc[h], 2);
    }
    float *pp = a.part_dr + (((size_t)tok * kTilesDN + tile) * kBlkDN + b) * 16;
    if (t == 0) {
        pp[g] = racc[0];
        pp[g + 8] = racc[1];
    }
    if (last_arrival(a.cnt_dn + tile, kBlkDN * (a.T + 1))) dn_finish(a, tile);
}

// One token's six routed experts, 16 rows x 256 cols each (Q2_K).
__device__ __forceinline__ void dn_routed_q2k(const DecodeArgs &a, const DNSmem &sm, long long r) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int tok = (int)(r / (kTilesDN * kBlkDN));
    const int rem = (int)(r % (kTilesDN * kBlkDN));
    const int tile = rem / kBlkDN, b = rem % kBlkDN;
    uint4 qa[kK], qb[kK];
    uint32_t sca[kK], scb[kK];
    uint2 dd[kK];
    bool ok[kK];
#pragma unroll
    for (int k = 0; k < kK; ++k) {
        const int e = a.ids[tok * kK + k];
        ok[k] = expert_ok(e, (const void *const *)a.down, nullptr, nullptr);
        if (ok[k]) {  // warp-uniform; an unusable id loads nothing
            const uint8_t *tb = a.down[e] + ((size_t)tile * kBlkDN + b) * kTB_Q2K;
            qa[k] = ldg_stream128(tb + 16 * lane);
            qb[k] = ldg_stream128(tb + 512 + 16 * lane);
            sca[k] = ldg_stream32(tb + 1024 + 4 * lane);
            scb[k] = ldg_stream32(tb + 1152 + 4 * lane);
            dd[k] = ldg_stream64(tb + 1280 + 8 * g);
        } else {
            qa[k] = qb[k] = make_uint4(0, 0, 0, 0);
            sca[k] = scb[k] = 0u;
            dd[k] = make_uint2(0, 0);
        }
    }
    const bool active = (g >> 1) == t;
    float racc[2] = {0.f, 0.f};
#pragma unroll
    for (int k = 0; k < kK; ++k) {
        const int slot = tok * kK + k;
        if (!ok[k]) {
            if (lane == 0) flag_status(a.status, DS4G_EDEVICE, (uint32_t)a.ids[slot]);
            continue;
        }
        const float wk = a.w[slot];
        const __half *hrow = sm.hq + ((size_t)slot * 2 + (g & 1)) * kF + 256 * b + 16 * t;
        const float4 X = *reinterpret_cast<const float4 *>(sm.xs + (size_t)slot * 128 + (b * 4 + t) * 4);
        const float4 S = *reinterpret_cast<const float4 *>(sm.hsc + (size_t)slot * 128 + (b * 4 + t) * 4);
        const float dg = __half2float(__ushort_as_half((unsigned short)(dd[k].x & 0xffff))) * 16777216.0f;
        const float mg = __half2float(__ushort_as_half((unsigned short)(dd[k].x >> 16)));
        const float dh = __half2float(__ushort_as_half((unsigned short)(dd[k].y & 0xffff))) * 16777216.0f;
        const float mh = __half2float(__ushort_as_half((unsigned short)(dd[k].y >> 16)));
        const uint32_t Wa[4] = {qa[k].x, qa[k].y, qa[k].z, qa[k].w};
        const uint32_t Wb[4] = {qb[k].x, qb[k].y, qb[k].z, qb[k].w};
        const float Xg[4] = {X.x, X.y, X.z, X.w};
        const float Sg[4] = {S.x, S.y, S.z, S.w};
        float sg = 0.f, sh = 0.f;
#pragma unroll
        for (int G = 0; G < 4; ++G) {
            float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const uint2 bv = active ? *reinterpret_cast<const uint2 *>(hrow + 64 * G + 4 * cc) : make_uint2(0, 0);
                mma_f16(c, (Wa[G] >> (4 * cc)) & 0x00030003u, (Wb[G] >> (4 * cc)) & 0x00030003u,
                        (Wa[G] >> (4 * cc + 2)) & 0x00030003u, (Wb[G] >> (4 * cc + 2)) & 0x00030003u, bv.x, bv.y);
            }
            const uint32_t ba = (sca[k] >> (8 * G)) & 0xffu, bb = (scb[k] >> (8 * G)) & 0xffu;
            sg += dg * small_u2f(ba & 15u) * ((c[0] + c[1]) * Sg[G]) - mg * small_u2f(ba >> 4) * Xg[G];
            sh += dh * small_u2f(bb & 15u) * ((c[2] + c[3]) * Sg[G]) - mh * small_u2f(bb >> 4) * Xg[G];
        }
        racc[0] = fmaf(wk, sg, racc[0]);
        racc[1] = fmaf(wk, sh, racc[1]);
    }
    dn_write_partial(a, tok, tile, b, racc);
}

// One token's six routed experts with Q4_K down (16 rows x 256 cols each).
__device__ __forceinline__ void dn_routed_q4k(const DecodeArgs &a, const DNSmem &sm, long long r) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int tok = (int)(r / (kTilesDN * kBlkDN));
    const int rem = (int)(r % (kTilesDN * kBlkDN));
    const int tile = rem / kBlkDN, b = rem % kBlkDN;
    const bool active = (g >> 1) == t;
    float racc[2] = {0.f, 0.f};
#pragma unroll 1
    for (int k = 0; k < kK; ++k) {
        const int slot = tok * kK + k;
        const int e = a.ids[slot];
        const bool ok = expert_ok(e, (const void *const *)a.down, nullptr, nullptr);
        if (!ok) {
            if (lane == 0) flag_status(a.status, DS4G_EDEVICE, (uint32_t)e);
            continue;
        }
        const uint8_t *tb = a.down[e] + ((size_t)tile * kBlkDN + b) * kTB_Q4K;
        uint4 q[2][2];
        uint32_t scw[2][3];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            q[h][0] = ldg_stream128(tb + 1024 * h + 32 * lane);
            q[h][1] = ldg_stream128(tb + 1024 * h + 32 * lane + 16);
#pragma unroll
            for (int i = 0; i < 3; ++i) scw[h][i] = ldg_stream32(tb + 2048 + 12 * (g + 8 * h) + 4 * i);
        }
        const uint2 dd = ldg_stream64(tb + 2240 + 8 * g);
        const float wk = a.w[slot];
        const float dgv[2] = {__half2float(__ushort_as_half((unsigned short)(dd.x & 0xffff))) * 16777216.0f,
                              __half2float(__ushort_as_half((unsigned short)(dd.y & 0xffff))) * 16777216.0f};
        const float dmv[2] = {__half2float(__ushort_as_half((unsigned short)(dd.x >> 16))),
                              __half2float(__ushort_as_half((unsigned short)(dd.y >> 16)))};
        const __half *hrow = sm.hq + ((size_t)slot * 2 + (g & 1)) * kF + 256 * b;
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            const int j = 4 * jj + t;  // 32-col sub-block = 16-col sub-blocks 2j, 2j+1
            const int ja = 2 * j, jb = 2 * j + 1;
            const int ia = (b * 4 + (ja & 3)) * 4 + (ja >> 2), ib = (b * 4 + (jb & 3)) * 4 + (jb >> 2);
            const float X = sm.xs[(size_t)slot * 128 + ia] + sm.xs[(size_t)slot * 128 + ib];
            const float Sa = sm.hsc[(size_t)slot * 128 + ia], Sb = sm.hsc[(size_t)slot * 128 + ib];
            // columns of the 16-entry groups ja (cc < 4) and jb (cc >= 4) of h
            // carry their own scales: one accumulator each
            float c[4] = {0.f, 0.f, 0.f, 0.f}, cb[4] = {0.f, 0.f, 0.f, 0.f};
            const uint32_t wa[4] = {q[0][jj].x, q[0][jj].y, q[0][jj].z, q[0][jj].w};
            const uint32_t wb[4] = {q[1][jj].x, q[1][jj].y, q[1][jj].z, q[1][jj].w};
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                const uint2 bv = active ? *reinterpret_cast<const uint2 *>(hrow + 32 * j + 4 * cc) : make_uint2(0, 0);
                const uint32_t Wa = wa[cc >> 1], Wb = wb[cc >> 1];
                const int s0 = 8 * (cc & 1);
                mma_f16(cc < 4 ? c : cb, (Wa >> s0) & 0x000F000Fu, (Wb >> s0) & 0x000F000Fu,
                        (Wa >> (s0 + 4)) & 0x000F000Fu, (Wb >> (s0 + 4)) & 0x000F000Fu, bv.x, bv.y);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t s0 = (scw[h][0] >> (8 * (j & 3))) & 0xffu;
                const uint32_t s1 = (scw[h][1] >> (8 * (j & 3))) & 0xffu;
                const uint32_t s2b = (scw[h][2] >> (8 * (j & 3))) & 0xffu;
                uint32_t sc, mn;
                if (j < 4) {
                    sc = s0 & 63u;
                    mn = s1 & 63u;
                } else {
                    sc = (s2b & 15u) | ((s0 >> 6) << 4);
                    mn = (s2b >> 4) | ((s1 >> 6) << 4);
                }
                const float dot = h ? (c[2] + c[3]) * Sa + (cb[2] + cb[3]) * Sb
                                    : (c[0] + c[1]) * Sa + (cb[0] + cb[1]) * Sb;
                racc[h] = fmaf(wk, dgv[h] * small_u2f(sc) * dot - dmv[h] * small_u2f(mn) * X, racc[h]);
            }
        }
    }
    dn_write_partial(a, tok, tile, b, racc);
}

// bf16 shared down task: 16 rows x 256 cols of Sd, all tokens.
__device__ __forceinline__ void dn_shared(const DecodeArgs &a, const DNSmem &sm, long long s) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int tile = (int)(s / kBlkDN), b = (int)(s % kBlkDN);
    uint2 A[16][2];
#pragma unroll
    for (int ch = 0; ch < 16; ++ch)
#pragma unroll
        for (int h = 0; h < 2; ++h)
            A[ch][h] = ldg_stream64(a.sh_down + (size_t)(tile * 16 + g + 8 * h) * kF + 256 * b + 16 * ch + 4 * t);
    const int tok = g >> 1;
    const bool has = tok < a.T;
    const __nv_bfloat16 *hrow = sm.hs + ((size_t)(has ? tok : 0) * 2 + (g & 1)) * kF + 256 * b + 4 * t;
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ch = 0; ch < 16; ++ch) {
        const uint2 bv = has ? *reinterpret_cast<const uint2 *>(hrow + 16 * ch) : make_uint2(0, 0);
        mma_bf16(c, A[ch][0].x, A[ch][1].x, A[ch][0].y, A[ch][1].y, bv.x, bv.y);
    }
    float *pp = a.part_ds + ((size_t)tile * kBlkDN + b) * a.T * 16;
    if (t < a.T) {
        pp[t * 16 + g] = c[0] + c[1];
        pp[t * 16 + g + 8] = c[2] + c[3];
    }
    if (last_arrival(a.cnt_dn + tile, kBlkDN * (a.T + 1))) dn_finish(a, tile);
}

__global__ void __launch_bounds__(kThreads, 1) down_decode_kernel(DecodeArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    DNSmem sm;
    const int nslot = kK * a.T;
    sm.hq = reinterpret_cast<__half *>(smem_raw);
    sm.xs = reinterpret_cast<float *>(sm.hq + (size_t)nslot * 2 * kF);
    sm.hsc = sm.xs + (size_t)nslot * 128;
    sm.hs = reinterpret_cast<__nv_bfloat16 *>(sm.hsc + (size_t)nslot * 128);
    const int tid = threadIdx.x;
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(a.hq);
        uint4 *dst = reinterpret_cast<uint4 *>(sm.hq);
        for (int i = tid; i < nslot * 2 * kF / 8; i += kThreads) dst[i] = __ldcg(src + i);
        const uint4 *s2 = reinterpret_cast<const uint4 *>(a.xs16);
        uint4 *d2 = reinterpret_cast<uint4 *>(sm.xs);
        for (int i = tid; i < nslot * 128 / 4; i += kThreads) d2[i] = __ldcg(s2 + i);
        const uint4 *s4 = reinterpret_cast<const uint4 *>(a.hsc16);
        uint4 *d4 = reinterpret_cast<uint4 *>(sm.hsc);
        for (int i = tid; i < nslot * 128 / 4; i += kThreads) d4[i] = __ldcg(s4 + i);
        const uint4 *s3 = reinterpret_cast<const uint4 *>(a.hs);
        uint4 *d3 = reinterpret_cast<uint4 *>(sm.hs);
        for (int i = tid; i < a.T * 2 * kF / 8; i += kThreads) d3[i] = __ldcg(s3 + i);
    }
    __syncthreads();
    const long long NR = (long long)a.T * kTilesDN * kBlkDN;
    const long long NS = (long long)kTilesDN * kBlkDN;
    const long long W = (long long)gridDim.x * kWarps;
    for (long long tau = blockIdx.x * kWarps + (tid >> 5); tau < NR + NS; tau += W) {
        long long idx;
        if (task_kind(tau, NR, NS, idx)) dn_shared(a, sm, idx);
        else if (a.dn_type == DS4G_Q2_K) dn_routed_q2k(a, sm, idx);
        else dn_routed_q4k(a, sm, idx);
    }
}

// ------------------------------------------------------------------ host
struct WsLayout {
    size_t cnt_gu, cnt_dn, part_r, part_s, hq, xs16, hsc16, hs, part_dr, part_ds, total;
};

// Tile counters at fixed offsets (sized for kDecodeMaxT tokens), scratch after.
static_assert(((size_t)kK * kDecodeMaxT + 1) * kTilesGU * 4 + (size_t)kTilesDN * 4 <= kWsDecCntBytes,
              "decode tile counters exceed their area");
static WsLayout ws_layout(int T) {
    const size_t ns = (size_t)kK * T;
    WsLayout L;
    L.cnt_gu = kWsDecCnt;
    L.cnt_dn = kWsDecCnt + ((size_t)kK * kDecodeMaxT + 1) * kTilesGU * 4;
    size_t off = kWsScratch;
    L.part_r = off;
    off += align_up(ns * kTilesGU * kSplitR * 32 * 4, 256);
    L.part_s = off;
    off += align_up((size_t)kTilesGU * kSplitS * 2 * T * 16 * 4, 256);
    L.hq = off;
    off += align_up(ns * 2 * kF * 2, 256);
    L.xs16 = off;
    off += align_up(ns * 128 * 4, 256);
    L.hsc16 = off;
    off += align_up(ns * 128 * 4, 256);
    L.hs = off;
    off += align_up((size_t)T * 2 * kF * 2, 256);
    L.part_dr = off;
    off += align_up((size_t)T * kTilesDN * kBlkDN * 16 * 4, 256);
    L.part_ds = off;
    off += align_up((size_t)kTilesDN * kBlkDN * T * 16 * 4, 256);
    L.total = off;
    return L;
}

size_t decode_workspace(int T) { return ws_layout(T).total; }

static int g_num_sms = 0;

ds4g_status decode_forward(const float *hidden, int T, const ds4g_layer *L, const int32_t *ids,
                           const float *w, float *out, void *workspace, cudaStream_t st, int phases,
                           uint32_t *status_word, const uint32_t *ready, uint32_t epoch, int q8) {
    if (!g_num_sms) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return DS4G_ECUDA;
        if (cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return DS4G_ECUDA;
    }
    DecodeArgs a;
    a.x = hidden;
    a.T = T;
    a.ids = ids;
    a.w = w;
    a.gu_type = L->gate_up_type;
    a.dn_type = L->down_type;
    a.gate = reinterpret_cast<const uint8_t *const *>(L->gate);
    a.up = reinterpret_cast<const uint8_t *const *>(L->up);
    a.down = reinterpret_cast<const uint8_t *const *>(L->down);
    a.sh_gate = reinterpret_cast<const __nv_bfloat16 *>(L->sh_gate);
    a.sh_up = reinterpret_cast<const __nv_bfloat16 *>(L->sh_up);
    a.sh_down = reinterpret_cast<const __nv_bfloat16 *>(L->sh_down);
    a.grid = L->iq2_grid;
    a.out = out;
    uint8_t *ws = (uint8_t *)workspace;
    const WsLayout wl = ws_layout(T);
    a.status = status_word ? status_word : (uint32_t *)ws;
    a.cnt_gu = (uint32_t *)(ws + wl.cnt_gu);
    a.cnt_dn = (uint32_t *)(ws + wl.cnt_dn);
    a.part_r = (float *)(ws + wl.part_r);
    a.part_s = (float *)(ws + wl.part_s);
    a.hq = (__half *)(ws + wl.hq);
    a.xs16 = (float *)(ws + wl.xs16);
    a.hsc16 = (float *)(ws + wl.hsc16);
    a.hs = (__nv_bfloat16 *)(ws + wl.hs);
    a.part_dr = (float *)(ws + wl.part_dr);
    a.part_ds = (float *)(ws + wl.part_ds);
    a.ready = ready;
    a.epoch = epoch;
    a.q8 = q8 && L->gate_up_type == DS4G_IQ2_XXS ? 1 : 0;

    const size_t ns = (size_t)kK * T;
    const size_t smem_gu = 256 * 16 * 8 + 128 * 16 * 8 + (size_t)T * 2 * kH * 2 * 2 +
                           (q8 ? 128 * 16 * 16 + (size_t)T * kH + (size_t)T * 16 * 4 : 0);
    const size_t smem_dn = ns * 2 * kF * 2 + 2 * ns * 128 * 4 + (size_t)T * 2 * kF * 2;
    static bool attr_done = false;
    if (!attr_done) {
        if (cudaFuncSetAttribute(gateup_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) !=
                cudaSuccess ||
            cudaFuncSetAttribute(down_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) !=
                cudaSuccess)
            return DS4G_ECUDA;
        attr_done = true;
    }
    if (phases & 1) {
        gateup_decode_kernel<<<g_num_sms, kThreads, smem_gu, st>>>(a);
        if (cudaGetLastError() != cudaSuccess) return DS4G_ECUDA;
    }
    if (phases & 2) {
        down_decode_kernel<<<g_num_sms, kThreads, smem_dn, st>>>(a);
        if (cudaGetLastError() != cudaSuccess) return DS4G_ECUDA;
    }
    return DS4G_OK;
}

}  // namespace ds4g
