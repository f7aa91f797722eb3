// batch.cu — the MoE block for a batch of 4..32 decode tokens (concurrent
// sessions decoded together), IQ2_XXS gate/up and Q2_K down (chenxutan ds4
// article §3.2: router result -> only the routed experts' weights -> shared
// expert -> merge; §3.3: only the selected experts are read).  The batch's
// 6T (token, slot) entries are grouped by expert, and every selected expert's
// packed tiles are read once per call and applied to all of its tokens.
//
//  bg_gateup_kernel  CTA c owns column quarter q = c % 4 of the 4096 inputs and
//      keeps the T tokens' activations for it in shared memory (fp16 hi, lo).
//      Warp tasks: (selected expert, 16-row tile, gate | up) over the quarter's
//      four tile-blocks, and (16-row tile, gate | up) of the shared expert.
//      Routed: exact codes on mma.sync with a block-diagonal activation (one
//      mma per token, the lane's own sub-block scales applied in fp32); the
//      operand registers of a grid row are built once and used for up to 4
//      tokens (a pass), with 4 / (tokens of the pass) independent accumulator
//      chains per token.  Shared: bf16 weights converted to fp16 (exact in the fp16
//      normal range), the tokens as the mma's N (8 per mma, hi and lo).
//      Output: per-quarter partial sums.
//  bg_h_kernel       h = silu(sum_q gate) * (sum_q up) per slot and row: routed
//      h as fp16 of 2^-e h (one power of two per 16 entries) with its
//      16-column sums and 2^e; shared h as fp16 hi, lo.
//  bg_down_kernel    CTA c owns 256-column block b = c % 8 of h and keeps it for
//      every slot in shared memory (routed: fp16 of 2^-e h; shared: hi, lo).
//      Warp tasks: (selected expert, two 16-row output tiles) over that
//      expert's slots, two slots per pass sharing each masked operand (Q2_K
//      quants exact, block-diagonal), and (16-row tile) of the
//      shared expert.  Output: per-block partials.
//  bg_combine_kernel out[t] = sum_b shared_b[t] + sum_k w[t,k] sum_b y_b[t,k],
//      in that fixed order.
// Slots whose expert id is out of range or whose matrices are missing add
// nothing and are flagged (DS4G_EDEVICE).
#include "ds4g_internal.cuh"

namespace ds4g {

constexpr int kBT = 32;                  // tokens per launch
constexpr int kBS = kBT * kK;            // slots per launch
constexpr int kBWarps = 16;
constexpr int kBThreads = kBWarps * 32;
constexpr int kBQ = 4;                   // column quarters of the gate/up input
constexpr int kBQC = kH / kBQ;           // 1024 columns per quarter
constexpr int kBXLd = kBQC + 8;          // fp16 row of a quarter (+16 B: no bank conflict)
constexpr int kBB = kF / 256;            // 256-column blocks of the down input
constexpr int kBHLd = 256 + 8;           // fp16 row of a block

struct BGArgs {
    const float *x;
    int T;
    const int32_t *ids;
    const float *w;
    const uint8_t *const *gate;
    const uint8_t *const *up;
    const uint8_t *const *down;
    const __nv_bfloat16 *sh_gate, *sh_up, *sh_down;
    const uint64_t *grid;
    float *out;
    uint32_t *status;
    float *P;       // [4 quarters][6T slots][2 gate, up][2048]
    float *PS;      // [4 quarters][T][2][2048]
    __half *hq;     // [6T][2048] fp16 of 2^-e h
    float *xs16;    // [6T][128] 16-column sums of h (permuted: (b*4 + j%4)*4 + j/4)
    float *hsc16;   // [6T][128] 2^e of each 16 entries (same layout)
    __half *hs;     // [T][2][2048] shared h, fp16 hi, lo
    float *Y;       // [8 blocks][6T][4096] routed down partials (unweighted)
    float *YS;      // [8 blocks][T][4096] shared down partials
};

// ------------------------------------------------------------ bucketing
// The batch's slots grouped by expert, in shared memory: experts in
// ascending id order, each with its slots in ascending (token, k) order.
struct BgBuckets {
    int ne;                  // distinct usable experts
    int16_t eid[kBS];        // expert of bucket i
    int16_t start[kBS + 1];  // bucket i's slots: slot[start[i] .. start[i+1])
    int16_t slot[kBS];
    int cnt[kE];
};

__device__ __forceinline__ bool bg_usable(const BGArgs &a, int e, bool gu) {
    return gu ? expert_ok(e, (const void *const *)a.gate, (const void *const *)a.up, nullptr)
              : expert_ok(e, (const void *const *)a.down, nullptr, nullptr);
}

// All threads of the CTA (>= 256).  gu: gate/up pointers checked, else down.
__device__ void bg_buckets(const BGArgs &a, BgBuckets &bk, bool gu) {
    const int tid = threadIdx.x, ns = kK * a.T;
    if (tid < kE) {
        int c = 0;
        for (int s = 0; s < ns; ++s) c += __ldg(a.ids + s) == tid;
        bk.cnt[tid] = (c && bg_usable(a, tid, gu)) ? c : 0;
    }
    if (tid < ns) {
        const int e = __ldg(a.ids + tid);
        if ((unsigned)e >= (unsigned)kE || !bg_usable(a, e, gu)) flag_status(a.status, DS4G_EDEVICE, (uint32_t)e);
    }
    __syncthreads();
    if (tid < 32) {
        // exclusive scans (8 experts per lane): slot offsets and bucket index
        int c[8], nz[8], sc = 0, sn = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            c[i] = bk.cnt[8 * tid + i];
            nz[i] = c[i] > 0;
            sc += c[i];
            sn += nz[i];
        }
        int ic = sc, in = sn;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, ic, o), v = __shfl_up_sync(0xffffffffu, in, o);
            if (tid >= o) {
                ic += u;
                in += v;
            }
        }
        int rc = ic - sc, rn = in - sn;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (nz[i]) {
                bk.eid[rn] = (int16_t)(8 * tid + i);
                bk.start[rn] = (int16_t)rc;
            }
            rc += c[i];
            rn += nz[i];
        }
        if (tid == 31) {
            bk.ne = rn;
            bk.start[rn] = (int16_t)rc;
        }
    }
    __syncthreads();
    if (tid < kE && bk.cnt[tid]) {
        // this expert's slots, in order (its bucket index: count of nonzero below it)
        int o = -1;
        for (int i = 0; i < bk.ne; ++i)
            if (bk.eid[i] == tid) o = bk.start[i];
        for (int s = 0; s < ns; ++s)
            if (__ldg(a.ids + s) == tid) bk.slot[o++] = (int16_t)s;
    }
    __syncthreads();
}

// ============================================================ gate / up
struct BgGuSmem {
    uint2 *gtab;     // [256][16] grid rows (value bytes), 16 replicas
    uint2 *stab;     // [128][16] sign bytes of each 7-bit sign index
    __half *x;       // [T][2][kBXLd] the quarter's activation, fp16 hi, lo
    BgBuckets *bk;
    int *next;       // the CTA's next unclaimed task
};

// One pass of bg_gu_routed over up to 4 of a bucket's slots (s0 ..): every
// grid row's operands are built once and multiplied by each token's
// block-diagonal activation.  NT = 1, 2 or 4 (3 and 4 tokens): each token
// accumulates into 4 / NT independent chains, so that few tokens still keep
// several MMAs in flight.
template <int NT>
__device__ __forceinline__ void bg_gu_pass(const BGArgs &a, const BgGuSmem &sm, const uint4 (&qa)[4],
                                           const uint4 (&qb)[4], const uint32_t (&dd)[4], int s0, int nt, int q,
                                           int rt, int m) {
    constexpr int CH = 4 / NT;   // accumulator chains per token
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3, p = lane & 15;
    const BgBuckets &bk = *sm.bk;
    const bool act = (g >> 1) == t;
    int tok[NT];
#pragma unroll
    for (int i = 0; i < NT; ++i) tok[i] = i < nt ? bk.slot[s0 + i] / kK : 0;
    float acc[NT][2];
#pragma unroll
    for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = 0.f;
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
        // d * 0.25 * 2^24 (the codes enter the mma as code * 2^-24)
        const float d4g = __half2float(__ushort_as_half((unsigned short)(dd[kb] & 0xffffu))) * 4194304.0f;
        const float d4h = __half2float(__ushort_as_half((unsigned short)(dd[kb] >> 16))) * 4194304.0f;
#pragma unroll 1
        for (int jj = 0; jj < 2; ++jj) {
            const uint32_t ia = jj ? qa[kb].z : qa[kb].x, va = jj ? qa[kb].w : qa[kb].y;
            const uint32_t ib = jj ? qb[kb].z : qb[kb].x, vb = jj ? qb[kb].w : qb[kb].y;
            float c[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i) c[i][0] = c[i][1] = c[i][2] = c[i][3] = 0.f;
#pragma unroll
            for (int l = 0; l < 4; ++l) {
                const uint2 ga = sm.gtab[((ia >> (8 * l)) & 255u) * 16 + p];
                const uint2 sa = sm.stab[((va >> (7 * l)) & 127u) * 16 + p];
                const uint2 gb = sm.gtab[((ib >> (8 * l)) & 255u) * 16 + p];
                const uint2 sbv = sm.stab[((vb >> (7 * l)) & 127u) * 16 + p];
                const uint32_t a0 = prmt(ga.x, sa.x, 0x5140), a1 = prmt(gb.x, sbv.x, 0x5140);
                const uint32_t a2 = prmt(ga.x, sa.x, 0x7362), a3 = prmt(gb.x, sbv.x, 0x7362);
                const uint32_t b0 = prmt(ga.y, sa.y, 0x5140), b1 = prmt(gb.y, sbv.y, 0x5140);
                const uint32_t b2 = prmt(ga.y, sa.y, 0x7362), b3 = prmt(gb.y, sbv.y, 0x7362);
                const int col = 256 * kb + 32 * (4 * jj + t) + 8 * l;
#pragma unroll
                for (int i = 0; i < NT; ++i) {
                    if (i < nt) {
                        uint4 B4 = make_uint4(0, 0, 0, 0);
                        if (act) B4 = *reinterpret_cast<const uint4 *>(sm.x + ((size_t)tok[i] * 2 + (g & 1)) * kBXLd + col);
                        mma_f16(c[i * CH + (2 * l) % CH], a0, a1, a2, a3, B4.x, B4.y);
                        mma_f16(c[i * CH + (2 * l + 1) % CH], b0, b1, b2, b3, B4.z, B4.w);
                    }
                }
            }
            const float sg = d4g * half_plus(va >> 28), sh = d4h * half_plus(vb >> 28);
#pragma unroll
            for (int i = 0; i < NT; ++i) {
                float u0 = 0.f, u1 = 0.f;
#pragma unroll
                for (int ch = 0; ch < CH; ++ch) {
                    u0 += c[i * CH + ch][0] + c[i * CH + ch][1];
                    u1 += c[i * CH + ch][2] + c[i * CH + ch][3];
                }
                acc[i][0] = fmaf(sg, u0, acc[i][0]);
                acc[i][1] = fmaf(sh, u1, acc[i][1]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < NT; ++i) {
        float r0 = acc[i][0], r1 = acc[i][1];
        r0 += __shfl_xor_sync(0xffffffffu, r0, 1);
        r0 += __shfl_xor_sync(0xffffffffu, r0, 2);
        r1 += __shfl_xor_sync(0xffffffffu, r1, 1);
        r1 += __shfl_xor_sync(0xffffffffu, r1, 2);
        if (i < nt && t == 0) {
            const int slot = bk.slot[s0 + i];
            float *pp = a.P + (((size_t)q * kK * a.T + slot) * 2 + m) * kF + 16 * rt;
            pp[g] = r0;
            pp[g + 8] = r1;
        }
    }
}

// A selected expert's gate or up rows 16 rt .. +16 over the CTA's quarter, for
// all slots of bucket bi (4 tokens per pass).  The quarter's four tile-blocks
// are loaded up front (four loads in flight per lane) and stay in registers
// across the passes; pf: the next task's tile-blocks, prefetched into L2.
__device__ __forceinline__ void bg_gu_routed(const BGArgs &a, const BgGuSmem &sm, int q, int bi, int rt, int m,
                                             const uint8_t *pf) {
    const int lane = threadIdx.x & 31, g = lane >> 2;
    const BgBuckets &bk = *sm.bk;
    const int e = bk.eid[bi];
    const uint8_t *tb0 = (m ? a.up[e] : a.gate[e]) + ((size_t)rt * 16 + 4 * q) * kTB_IQ2;
    uint4 qa[4], qb[4];
    uint32_t dd[4];
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
        qa[kb] = ldg_stream128(tb0 + kb * kTB_IQ2 + 16 * lane);
        qb[kb] = ldg_stream128(tb0 + kb * kTB_IQ2 + 512 + 16 * lane);
        dd[kb] = ldg_stream32(tb0 + kb * kTB_IQ2 + 1024 + 4 * g);
    }
    if (pf) asm volatile("prefetch.global.L2 [%0];" ::"l"(pf + 128 * lane));   // 4 tile-blocks = 4224 B
    for (int s0 = bk.start[bi]; s0 < bk.start[bi + 1]; s0 += 4) {
        const int nt = min(4, bk.start[bi + 1] - s0);
        // fewer tokens, more independent accumulator chains per token
        if (nt == 1) bg_gu_pass<1>(a, sm, qa, qb, dd, s0, nt, q, rt, m);
        else if (nt == 2) bg_gu_pass<2>(a, sm, qa, qb, dd, s0, nt, q, rt, m);
        else bg_gu_pass<4>(a, sm, qa, qb, dd, s0, nt, q, rt, m);
    }
}

// Two bf16 weights (one 32-bit word) -> two fp16 (one word); exact for
// weights in the fp16 normal range (the bf16 value has 8 significant bits).
__device__ __forceinline__ uint32_t bf2h2(uint32_t v) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(__uint_as_float(v & 0xffff0000u)), "f"(__uint_as_float(v << 16)));
    return r;
}

// The shared expert's gate or up rows 16 rt .. +16 over the CTA's quarter,
// all tokens (the tokens as the mma's N: 8 per mma, hi and lo).  Inside each
// 64-column chunk lane t takes columns 16t .. 16t+15 (k-slice s: 16t + 4s ..
// +3), the same permutation on both operands.
__device__ __forceinline__ void bg_gu_shared(const BGArgs &a, const BgGuSmem &sm, int q, int rt, int m) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const __nv_bfloat16 *W = (m ? a.sh_up : a.sh_gate) + (size_t)(16 * rt + g) * kH + kBQC * q + 16 * t;
    const int ngr = (a.T + 7) / 8;
    float c[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i][0] = c[i][1] = c[i][2] = c[i][3] = 0.f;
    // chunk ch + 1 loads while chunk ch is multiplied
    uint4 na0 = ldg_stream128(W), na1 = ldg_stream128(W + 8);
    uint4 nb0 = ldg_stream128(W + 8 * kH), nb1 = ldg_stream128(W + 8 * kH + 8);
#pragma unroll 1
    for (int ch = 0; ch < kBQC / 64; ++ch) {
        const uint4 ra0 = na0, ra1 = na1, rb0 = nb0, rb1 = nb1;
        if (ch + 1 < kBQC / 64) {
            na0 = ldg_stream128(W + 64 * (ch + 1));
            na1 = ldg_stream128(W + 64 * (ch + 1) + 8);
            nb0 = ldg_stream128(W + 8 * kH + 64 * (ch + 1));
            nb1 = ldg_stream128(W + 8 * kH + 64 * (ch + 1) + 8);
        }
        const uint32_t A[8] = {bf2h2(ra0.x), bf2h2(ra0.y), bf2h2(ra0.z), bf2h2(ra0.w),
                               bf2h2(ra1.x), bf2h2(ra1.y), bf2h2(ra1.z), bf2h2(ra1.w)};
        const uint32_t Bw[8] = {bf2h2(rb0.x), bf2h2(rb0.y), bf2h2(rb0.z), bf2h2(rb0.w),
                                bf2h2(rb1.x), bf2h2(rb1.y), bf2h2(rb1.z), bf2h2(rb1.w)};
#pragma unroll
        for (int gr = 0; gr < 4; ++gr) {
            if (gr >= ngr) break;
            const int tk = 8 * gr + g;
            const bool has = tk < a.T;
            const __half *xr = sm.x + ((size_t)(has ? tk : 0) * 2) * kBXLd + 64 * ch + 16 * t;
#pragma unroll
            for (int hl = 0; hl < 2; ++hl) {
                uint4 x0 = make_uint4(0, 0, 0, 0), x1 = make_uint4(0, 0, 0, 0);
                if (has) {
                    x0 = *reinterpret_cast<const uint4 *>(xr + hl * kBXLd);
                    x1 = *reinterpret_cast<const uint4 *>(xr + hl * kBXLd + 8);
                }
                const uint32_t X[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                for (int s = 0; s < 4; ++s) mma_f16(c[gr], A[2 * s], Bw[2 * s], A[2 * s + 1], Bw[2 * s + 1], X[2 * s], X[2 * s + 1]);
            }
        }
    }
#pragma unroll
    for (int gr = 0; gr < 4; ++gr) {
        if (gr >= ngr) break;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int tk = 8 * gr + 2 * t + j;
            if (tk < a.T) {
                float *pp = a.PS + (((size_t)q * a.T + tk) * 2 + m) * kF + 16 * rt;
                pp[g] = c[gr][j];
                pp[g + 8] = c[gr][2 + j];
            }
        }
    }
}

__global__ void __launch_bounds__(kBThreads, 1) bg_gateup_kernel(BGArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    BgGuSmem sm;
    sm.gtab = reinterpret_cast<uint2 *>(smem_raw);
    sm.stab = sm.gtab + 256 * 16;
    sm.x = reinterpret_cast<__half *>(sm.stab + 128 * 16);
    sm.bk = reinterpret_cast<BgBuckets *>(sm.x + (size_t)a.T * 2 * kBXLd);
    sm.next = reinterpret_cast<int *>(sm.bk + 1);
    const int tid = threadIdx.x;
    const int q = blockIdx.x % kBQ, ci = blockIdx.x / kBQ;
    const int ncq = (gridDim.x - q + kBQ - 1) / kBQ;   // CTAs of this quarter
    for (int i = tid; i < 256 * 16; i += kBThreads) {
        const uint64_t row = a.grid[i >> 4];
        sm.gtab[i] = make_uint2((uint32_t)row, (uint32_t)(row >> 32));
    }
    for (int i = tid; i < 128 * 16; i += kBThreads) {
        const uint32_t s7 = (uint32_t)(i >> 4);
        const uint32_t sg = s7 | ((uint32_t)(__popc(s7) & 1) << 7);
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            lo |= ((sg >> j) & 1u) << (8 * j + 7);
            hi |= ((sg >> (j + 4)) & 1u) << (8 * j + 7);
        }
        sm.stab[i] = make_uint2(lo, hi);
    }
    for (int i = tid; i < a.T * kBQC; i += kBThreads) {
        const int tk = i / kBQC, c = i % kBQC;
        const float v = a.x[(size_t)tk * kH + kBQC * q + c];
        if (!(fabsf(v) < 65504.f)) flag_status(a.status, DS4G_EDEVICE, 0xF16u);
        __half hi, lo;
        split_f16(v, hi, lo);
        sm.x[((size_t)tk * 2) * kBXLd + c] = hi;
        sm.x[((size_t)tk * 2 + 1) * kBXLd + c] = lo;
    }
    if (tid == 0) *sm.next = 0;
    bg_buckets(a, *sm.bk, true);   // ends with __syncthreads
    // tasks of this quarter: 256 shared (tile, matrix), then per bucket 256
    // routed (tile, matrix); task i of the quarter goes to CTA i % ncq
    const int nshared = (kF / 16) * 2, ntask = nshared + sm.bk->ne * (kF / 16) * 2;
    const int nmine = ntask > ci ? (ntask - ci + ncq - 1) / ncq : 0;
    // the warp claims its next task one ahead, so that task's weights can be
    // prefetched into L2 while the current one runs
    int k = 0;
    if ((tid & 31) == 0) k = atomicAdd(sm.next, 1);
    k = __shfl_sync(0xffffffffu, k, 0);
    while (k < nmine) {
        int kn = 0;
        if ((tid & 31) == 0) kn = atomicAdd(sm.next, 1);
        kn = __shfl_sync(0xffffffffu, kn, 0);
        const int task = ci + k * ncq;
        if (task < nshared) {
            bg_gu_shared(a, sm, q, task >> 1, task & 1);
        } else {
            const int r = task - nshared;
            const uint8_t *pf = nullptr;
            const int taskn = ci + kn * ncq;
            if (kn < nmine && taskn >= nshared) {
                const int rn = taskn - nshared, bn = rn / ((kF / 16) * 2);
                const int en = sm.bk->eid[bn];
                pf = ((rn & 1) ? a.up[en] : a.gate[en]) + ((size_t)((rn >> 1) % (kF / 16)) * 16 + 4 * q) * kTB_IQ2;
            }
            bg_gu_routed(a, sm, q, r / ((kF / 16) * 2), (r >> 1) % (kF / 16), r & 1, pf);
        }
        k = kn;
    }
}

// ================================================================= h
// One warp per (row of slots and shared tokens, 16-row group).
__global__ void __launch_bounds__(256) bg_h_kernel(BGArgs a) {
    const int lane = threadIdx.x & 31;
    const int wid = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int nrow = kK * a.T + a.T;
    if (wid >= nrow * (kF / 16)) return;
    const int r = wid / (kF / 16), j = wid % (kF / 16);
    const int row = 16 * j + (lane & 15);
    float gs = 0.f, us = 0.f;
    const bool routed = r < kK * a.T;
    if (lane < 16) {
#pragma unroll
        for (int q = 0; q < kBQ; ++q) {
            const float *pp = routed ? a.P + (((size_t)q * kK * a.T + r) * 2) * kF
                                     : a.PS + (((size_t)q * a.T + (r - kK * a.T)) * 2) * kF;
            gs += __ldcg(pp + row);
            us += __ldcg(pp + kF + row);
        }
    }
    const float hv = lane < 16 ? silu_f(gs) * us : 0.f;
    if (routed) {
        const int e = a.ids[r];
        const bool ok = expert_ok(e, (const void *const *)a.gate, (const void *const *)a.up,
                                  (const void *const *)a.down);
        float h = ok ? hv : 0.f;
        if (lane < 16 && !(fabsf(h) <= 3.4028235e38f)) flag_status(a.status, DS4G_EDEVICE, 0xF16u);
        float sum = h, mx = fabsf(h);
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) {
            sum += __shfl_xor_sync(0xffffffffu, sum, o);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        const int ex = h_group_exp(mx);
        if (lane < 16) a.hq[(size_t)r * kF + row] = __float2half_rn(h * pow2f(-ex));
        if (lane == 0) {
            const int b = j >> 4, j16 = j & 15;
            a.xs16[(size_t)r * 128 + (b * 4 + (j16 & 3)) * 4 + (j16 >> 2)] = sum;
            a.hsc16[(size_t)r * 128 + (b * 4 + (j16 & 3)) * 4 + (j16 >> 2)] = pow2f(ex);
        }
    } else if (lane < 16) {
        if (!(fabsf(hv) < 65504.f)) flag_status(a.status, DS4G_EDEVICE, 0xF16u);
        __half hi, lo;
        split_f16(hv, hi, lo);
        const int tk = r - kK * a.T;
        a.hs[((size_t)tk * 2) * kF + row] = hi;
        a.hs[((size_t)tk * 2 + 1) * kF + row] = lo;
    }
}

// ================================================================= down
struct BgDnSmem {
    __half *h;       // [6T][kBHLd] block b of 2^-e h (routed slots)
    float *xs;       // [6T][16] 16-column sums of h for block b
    float *hsc;      // [6T][16] 2^e for block b
    __half *hs;      // [T][2][kBHLd] block b of the shared h, hi, lo
    BgBuckets *bk;
    int *next;
};

// (x >> sh) & m, recomputed where it is used: keeps the compiler from hoisting every
// masked operand of four tile-blocks out of the slot loop (256 registers).
__device__ __forceinline__ uint32_t and_here(uint32_t x, uint32_t sh, uint32_t m) {
    uint32_t r;
    asm volatile("{\n\t.reg .b32 u;\n\tshr.b32 u, %1, %2;\n\tand.b32 %0, u, %3;\n\t}" : "=r"(r) : "r"(x), "r"(sh), "r"(m));
    return r;
}

// One pass of bg_dn_routed over up to NS of a bucket's slots (s0 ..): each
// masked Q2_K operand of the two tile-blocks is built once per pass and
// multiplied by every slot's block-diagonal h; per slot the arithmetic (mma
// chain over cc, then the scale and min terms, summed over G in order) is
// the same as for a single slot.
template <int NS>
__device__ __forceinline__ void bg_dn_pass(const BGArgs &a, const BgDnSmem &sm, int b, int og, const uint4 (&qa)[2],
                                           const uint4 (&qb)[2], const uint32_t (&sca)[2], const uint32_t (&scb)[2],
                                           const uint2 (&dd)[2], int s0, int ns) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const BgBuckets &bk = *sm.bk;
    // B: h of the slot (the lanes with g == 2t; column 2t + 1 of B stays zero)
    const bool act = g == 2 * t;
    int slot[NS];
    float4 X[NS], S[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i) {
        slot[i] = bk.slot[s0 + (i < ns ? i : 0)];
        X[i] = *reinterpret_cast<const float4 *>(sm.xs + (size_t)slot[i] * 16 + 4 * t);
        S[i] = *reinterpret_cast<const float4 *>(sm.hsc + (size_t)slot[i] * 16 + 4 * t);
    }
    float dg[2], mg[2], dh[2], mh[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        dg[u] = __half2float(__ushort_as_half((unsigned short)(dd[u].x & 0xffff))) * 16777216.0f;
        mg[u] = __half2float(__ushort_as_half((unsigned short)(dd[u].x >> 16)));
        dh[u] = __half2float(__ushort_as_half((unsigned short)(dd[u].y & 0xffff))) * 16777216.0f;
        mh[u] = __half2float(__ushort_as_half((unsigned short)(dd[u].y >> 16)));
    }
    float sg[NS][2], sh[NS][2];
#pragma unroll
    for (int i = 0; i < NS; ++i) sg[i][0] = sg[i][1] = sh[i][0] = sh[i][1] = 0.f;
#pragma unroll
    for (int G = 0; G < 4; ++G) {
        uint2 hv[NS][4];
#pragma unroll
        for (int i = 0; i < NS; ++i) {
            const __half *hrow = sm.h + (size_t)slot[i] * kBHLd + 16 * t + 64 * G;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
                hv[i][cc] = act ? *reinterpret_cast<const uint2 *>(hrow + 4 * cc) : make_uint2(0, 0);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const uint32_t Wa = G == 0 ? qa[u].x : G == 1 ? qa[u].y : G == 2 ? qa[u].z : qa[u].w;
            const uint32_t Wb = G == 0 ? qb[u].x : G == 1 ? qb[u].y : G == 2 ? qb[u].z : qb[u].w;
            uint32_t op[4][4];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                op[cc][0] = and_here(Wa, 4 * cc, 0x00030003u);
                op[cc][1] = and_here(Wb, 4 * cc, 0x00030003u);
                op[cc][2] = and_here(Wa, 4 * cc + 2, 0x00030003u);
                op[cc][3] = and_here(Wb, 4 * cc + 2, 0x00030003u);
            }
            const uint32_t ba = (sca[u] >> (8 * G)) & 0xffu, bb = (scb[u] >> (8 * G)) & 0xffu;
            const float kg = dg[u] * small_u2f(ba & 15u), ng = mg[u] * small_u2f(ba >> 4);
            const float kh = dh[u] * small_u2f(bb & 15u), nh = mh[u] * small_u2f(bb >> 4);
#pragma unroll
            for (int i = 0; i < NS; ++i) {
                if (i < ns) {
                    const float Xg = G == 0 ? X[i].x : G == 1 ? X[i].y : G == 2 ? X[i].z : X[i].w;
                    const float Sg = G == 0 ? S[i].x : G == 1 ? S[i].y : G == 2 ? S[i].z : S[i].w;
                    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
                        mma_f16(c, op[cc][0], op[cc][1], op[cc][2], op[cc][3], hv[i][cc].x, hv[i][cc].y);
                    sg[i][u] += kg * ((c[0] + c[1]) * Sg) - ng * Xg;
                    sh[i][u] += kh * ((c[2] + c[3]) * Sg) - nh * Xg;
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < NS; ++i) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            float r0 = sg[i][u], r1 = sh[i][u];
            r0 += __shfl_xor_sync(0xffffffffu, r0, 1);
            r0 += __shfl_xor_sync(0xffffffffu, r0, 2);
            r1 += __shfl_xor_sync(0xffffffffu, r1, 1);
            r1 += __shfl_xor_sync(0xffffffffu, r1, 2);
            if (i < ns && t == 0) {
                float *yy = a.Y + ((size_t)b * kK * a.T + slot[i]) * kH + 16 * (2 * og + u);
                yy[g] = r0;
                yy[g + 8] = r1;
            }
        }
    }
}

// A selected expert's Q2_K down rows 32 og .. +32 (two 16-row tiles), block
// b of h, for all slots of bucket bi (two slots per pass).  The two
// tile-blocks are loaded up front and stay in registers across the passes;
// pf: the warp's next task's tile-blocks, prefetched into L2.
__device__ __forceinline__ void bg_dn_routed(const BGArgs &a, const BgDnSmem &sm, int b, int bi, int og,
                                             const uint8_t *pf) {
    const int lane = threadIdx.x & 31, g = lane >> 2;
    const BgBuckets &bk = *sm.bk;
    const int e = bk.eid[bi];
    uint4 qa[2], qb[2];
    uint32_t sca[2], scb[2];
    uint2 dd[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const uint8_t *tb = a.down[e] + ((size_t)(2 * og + u) * kBB + b) * kTB_Q2K;
        qa[u] = ldg_stream128(tb + 16 * lane);
        qb[u] = ldg_stream128(tb + 512 + 16 * lane);
        sca[u] = ldg_stream32(tb + 1024 + 4 * lane);
        scb[u] = ldg_stream32(tb + 1152 + 4 * lane);
        dd[u] = ldg_stream64(tb + 1280 + 8 * g);
    }
    // lanes 0..10: the first tile-block (1344 B), lanes 16..26: the second
    if (pf && (lane & 15) < 11)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(pf + (size_t)(lane >> 4) * kBB * kTB_Q2K + 128 * (lane & 15)));
    for (int s0 = bk.start[bi]; s0 < bk.start[bi + 1]; s0 += 2) {
        const int ns = min(2, bk.start[bi + 1] - s0);
        if (ns == 1) bg_dn_pass<1>(a, sm, b, og, qa, qb, sca, scb, dd, s0, ns);
        else bg_dn_pass<2>(a, sm, b, og, qa, qb, sca, scb, dd, s0, ns);
    }
}

// The shared expert's down rows 16 ot .. +16, block b, all tokens (tokens as N).
__device__ __forceinline__ void bg_dn_shared(const BGArgs &a, const BgDnSmem &sm, int b, int ot) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const __nv_bfloat16 *W = a.sh_down + (size_t)(16 * ot + g) * kF + 256 * b + 16 * t;
    const int ngr = (a.T + 7) / 8;
    float c[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i][0] = c[i][1] = c[i][2] = c[i][3] = 0.f;
    // chunk ch + 1 loads while chunk ch is multiplied
    uint4 na0 = ldg_stream128(W), na1 = ldg_stream128(W + 8);
    uint4 nb0 = ldg_stream128(W + 8 * kF), nb1 = ldg_stream128(W + 8 * kF + 8);
#pragma unroll 1
    for (int ch = 0; ch < 4; ++ch) {
        const uint4 ra0 = na0, ra1 = na1, rb0 = nb0, rb1 = nb1;
        if (ch + 1 < 4) {
            na0 = ldg_stream128(W + 64 * (ch + 1));
            na1 = ldg_stream128(W + 64 * (ch + 1) + 8);
            nb0 = ldg_stream128(W + 8 * kF + 64 * (ch + 1));
            nb1 = ldg_stream128(W + 8 * kF + 64 * (ch + 1) + 8);
        }
        const uint32_t A[8] = {bf2h2(ra0.x), bf2h2(ra0.y), bf2h2(ra0.z), bf2h2(ra0.w),
                               bf2h2(ra1.x), bf2h2(ra1.y), bf2h2(ra1.z), bf2h2(ra1.w)};
        const uint32_t Bw[8] = {bf2h2(rb0.x), bf2h2(rb0.y), bf2h2(rb0.z), bf2h2(rb0.w),
                                bf2h2(rb1.x), bf2h2(rb1.y), bf2h2(rb1.z), bf2h2(rb1.w)};
#pragma unroll
        for (int gr = 0; gr < 4; ++gr) {
            if (gr >= ngr) break;
            const int tk = 8 * gr + g;
            const bool has = tk < a.T;
            const __half *hr = sm.hs + ((size_t)(has ? tk : 0) * 2) * kBHLd + 64 * ch + 16 * t;
#pragma unroll
            for (int hl = 0; hl < 2; ++hl) {
                uint4 x0 = make_uint4(0, 0, 0, 0), x1 = make_uint4(0, 0, 0, 0);
                if (has) {
                    x0 = *reinterpret_cast<const uint4 *>(hr + hl * kBHLd);
                    x1 = *reinterpret_cast<const uint4 *>(hr + hl * kBHLd + 8);
                }
                const uint32_t X[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                for (int s = 0; s < 4; ++s) mma_f16(c[gr], A[2 * s], Bw[2 * s], A[2 * s + 1], Bw[2 * s + 1], X[2 * s], X[2 * s + 1]);
            }
        }
    }
#pragma unroll
    for (int gr = 0; gr < 4; ++gr) {
        if (gr >= ngr) break;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int tk = 8 * gr + 2 * t + j;
            if (tk < a.T) {
                float *yy = a.YS + ((size_t)b * a.T + tk) * kH + 16 * ot;
                yy[g] = c[gr][j];
                yy[g + 8] = c[gr][2 + j];
            }
        }
    }
}

__global__ void __launch_bounds__(kBThreads, 1) bg_down_kernel(BGArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    BgDnSmem sm;
    const int ns = kK * a.T;
    sm.h = reinterpret_cast<__half *>(smem_raw);
    sm.xs = reinterpret_cast<float *>(sm.h + (size_t)ns * kBHLd);
    sm.hsc = sm.xs + (size_t)ns * 16;
    sm.hs = reinterpret_cast<__half *>(sm.hsc + (size_t)ns * 16);
    sm.bk = reinterpret_cast<BgBuckets *>(sm.hs + (size_t)a.T * 2 * kBHLd);
    sm.next = reinterpret_cast<int *>(sm.bk + 1);
    const int tid = threadIdx.x;
    const int b = blockIdx.x % kBB, ci = blockIdx.x / kBB;
    const int ncb = (gridDim.x - b + kBB - 1) / kBB;
    // block b of every slot's h (and its sums and scales), of the shared h
    for (int i = tid; i < ns * 32; i += kBThreads) {
        const int s = i >> 5, c8 = i & 31;
        *reinterpret_cast<uint4 *>(sm.h + (size_t)s * kBHLd + 8 * c8) =
            __ldcg(reinterpret_cast<const uint4 *>(a.hq + (size_t)s * kF + 256 * b) + c8);
    }
    for (int i = tid; i < ns * 16; i += kBThreads) {
        const int s = i >> 4, k = i & 15;
        sm.xs[i] = __ldcg(a.xs16 + (size_t)s * 128 + 16 * b + k);
        sm.hsc[i] = __ldcg(a.hsc16 + (size_t)s * 128 + 16 * b + k);
    }
    for (int i = tid; i < a.T * 2 * 32; i += kBThreads) {
        const int r = i >> 5, c8 = i & 31;
        *reinterpret_cast<uint4 *>(sm.hs + (size_t)r * kBHLd + 8 * c8) =
            __ldcg(reinterpret_cast<const uint4 *>(a.hs + (size_t)r * kF + 256 * b) + c8);
    }
    if (tid == 0) *sm.next = 0;
    bg_buckets(a, *sm.bk, false);   // ends with __syncthreads
    // tasks: 256 shared (16-row tile), then per bucket 128 routed (two tiles)
    const int nshared = kH / 16, ntask = nshared + sm.bk->ne * (kH / 32);
    const int nmine = ntask > ci ? (ntask - ci + ncb - 1) / ncb : 0;
    // the warp claims its next task one ahead, so that task's weights can be
    // prefetched into L2 while the current one runs
    int k = 0;
    if ((tid & 31) == 0) k = atomicAdd(sm.next, 1);
    k = __shfl_sync(0xffffffffu, k, 0);
    while (k < nmine) {
        int kn = 0;
        if ((tid & 31) == 0) kn = atomicAdd(sm.next, 1);
        kn = __shfl_sync(0xffffffffu, kn, 0);
        const int task = ci + k * ncb;
        if (task < nshared) {
            bg_dn_shared(a, sm, b, task);
        } else {
            const uint8_t *pf = nullptr;
            const int taskn = ci + kn * ncb;
            if (kn < nmine && taskn >= nshared) {
                const int rn = taskn - nshared;
                pf = a.down[sm.bk->eid[rn / (kH / 32)]] + ((size_t)(2 * (rn % (kH / 32))) * kBB + b) * kTB_Q2K;
            }
            bg_dn_routed(a, sm, b, (task - nshared) / (kH / 32), (task - nshared) % (kH / 32), pf);
        }
        k = kn;
    }
}

// ============================================================== combine
// out[t][r] = sum_b YS[b][t][r] + sum_k w[t,k] * sum_b Y[b][6t+k][r], fixed order.
__global__ void __launch_bounds__(256) bg_combine_kernel(BGArgs a) {
    const int t = blockIdx.y, r = 256 * blockIdx.x + threadIdx.x;
    float v = 0.f;
    for (int b = 0; b < kBB; ++b) v += __ldcs(a.YS + ((size_t)b * a.T + t) * kH + r);
    for (int k = 0; k < kK; ++k) {
        const int slot = kK * t + k;
        const int e = a.ids[slot];
        if (!expert_ok(e, (const void *const *)a.gate, (const void *const *)a.up, (const void *const *)a.down)) continue;
        float y = 0.f;
        for (int b = 0; b < kBB; ++b) y += __ldcs(a.Y + ((size_t)b * kK * a.T + slot) * kH + r);
        v = fmaf(a.w[slot], y, v);
    }
    a.out[(size_t)t * kH + r] = v;
}

// ------------------------------------------------------------------ host
struct BgLayout {
    size_t P, PS, hq, xs16, hsc16, hs, Y, YS, total;
};

static BgLayout bg_layout(int T) {
    const size_t ns = (size_t)kK * T;
    BgLayout L;
    size_t off = kWsScratch;
    L.P = off;
    off += align_up(kBQ * ns * 2 * kF * 4, 256);
    L.PS = off;
    off += align_up((size_t)kBQ * T * 2 * kF * 4, 256);
    L.hq = off;
    off += align_up(ns * kF * 2, 256);
    L.xs16 = off;
    off += align_up(ns * 128 * 4, 256);
    L.hsc16 = off;
    off += align_up(ns * 128 * 4, 256);
    L.hs = off;
    off += align_up((size_t)T * 2 * kF * 2, 256);
    L.Y = off;
    off += align_up((size_t)kBB * ns * kH * 4, 256);
    L.YS = off;
    off += align_up((size_t)kBB * T * kH * 4, 256);
    L.total = off;
    return L;
}

size_t batch_workspace(int T) { return bg_layout(T < kBT ? T : kBT).total; }

static size_t bg_gu_smem(int T) {
    return 256 * 16 * 8 + 128 * 16 * 8 + (size_t)T * 2 * kBXLd * 2 + sizeof(BgBuckets) + 16;
}
static size_t bg_dn_smem(int T) {
    return (size_t)kK * T * kBHLd * 2 + 2 * (size_t)kK * T * 16 * 4 + (size_t)T * 2 * kBHLd * 2 +
           sizeof(BgBuckets) + 16;
}

static int g_bg_sms = 0;
static bool g_bg_attr = false;

// One launch group for up to kBT tokens.
static ds4g_status batch_chunk(const float *hidden, int T, const ds4g_layer *L, const int32_t *ids, const float *w,
                               float *out, void *workspace, cudaStream_t st) {
    BGArgs a;
    a.x = hidden;
    a.T = T;
    a.ids = ids;
    a.w = w;
    a.gate = reinterpret_cast<const uint8_t *const *>(L->gate);
    a.up = reinterpret_cast<const uint8_t *const *>(L->up);
    a.down = reinterpret_cast<const uint8_t *const *>(L->down);
    a.sh_gate = reinterpret_cast<const __nv_bfloat16 *>(L->sh_gate);
    a.sh_up = reinterpret_cast<const __nv_bfloat16 *>(L->sh_up);
    a.sh_down = reinterpret_cast<const __nv_bfloat16 *>(L->sh_down);
    a.grid = L->iq2_grid;
    a.out = out;
    uint8_t *ws = (uint8_t *)workspace;
    const BgLayout wl = bg_layout(T);
    a.status = (uint32_t *)ws;
    a.P = (float *)(ws + wl.P);
    a.PS = (float *)(ws + wl.PS);
    a.hq = (__half *)(ws + wl.hq);
    a.xs16 = (float *)(ws + wl.xs16);
    a.hsc16 = (float *)(ws + wl.hsc16);
    a.hs = (__half *)(ws + wl.hs);
    a.Y = (float *)(ws + wl.Y);
    a.YS = (float *)(ws + wl.YS);
    bg_gateup_kernel<<<g_bg_sms, kBThreads, bg_gu_smem(T), st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return DS4G_ECUDA;
    const int nw = (kK * T + T) * (kF / 16);
    bg_h_kernel<<<(nw + 7) / 8, 256, 0, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return DS4G_ECUDA;
    bg_down_kernel<<<g_bg_sms, kBThreads, bg_dn_smem(T), st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return DS4G_ECUDA;
    bg_combine_kernel<<<dim3(kH / 256, T), 256, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? DS4G_OK : DS4G_ECUDA;
}

// The batched path for 4 <= T < 64 (IQ2_XXS gate/up, Q2_K down): chunks of
// up to 32 tokens.
ds4g_status batch_forward(const float *hidden, int T, const ds4g_layer *L, const int32_t *ids, const float *w,
                          float *out, void *workspace, cudaStream_t st) {
    if (!g_bg_sms) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return DS4G_ECUDA;
        if (cudaDeviceGetAttribute(&g_bg_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return DS4G_ECUDA;
    }
    if (!g_bg_attr) {
        if (cudaFuncSetAttribute(bg_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)bg_gu_smem(kBT)) != cudaSuccess ||
            cudaFuncSetAttribute(bg_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)bg_dn_smem(kBT)) != cudaSuccess)
            return DS4G_ECUDA;
        g_bg_attr = true;
    }
    for (int t0 = 0; t0 < T; t0 += kBT) {
        const int n = T - t0 < kBT ? T - t0 : kBT;
        const ds4g_status rc = batch_chunk(hidden + (size_t)t0 * kH, n, L, ids + (size_t)t0 * kK,
                                           w + (size_t)t0 * kK, out + (size_t)t0 * kH, workspace, st);
        if (rc != DS4G_OK) return rc;
    }
    return DS4G_OK;
}

}  // namespace ds4g
