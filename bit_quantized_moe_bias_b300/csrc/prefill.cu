// prefill.cu — the MoE block for many tokens at once (chunked prefill,
// chenxutan ds4 article §2.3; the block per §3.2: router result -> only the
// routed experts -> shared expert -> merge; formats of the juejin ds4 article
// §2.3).  The routed experts become a grouped GEMM over token buckets, the one
// dense contraction of the block, on the 5th-generation tensor cores:
//
//   bucket   counts / offsets / perm / inv of the 6T (token, slot) entries
//   permute  xb[slot] = bf16(x[token of slot]) for the 6T slots, then the T
//            tokens in order (rows 6T..7T-1, the shared expert's operand)
//   gate/up  per (group, 128-row tile of G/U, chunk of <= 128 bucket rows):
//            D_g = G_tile . xb_rows^T, D_u = U_tile . xb_rows^T in TMEM,
//            epilogue h = silu(D_g) * D_u -> h32 (fp32)
//   cast     per row of h32: routed rows -> fp16 of 2^-e h with one power of
//            two 2^e per row (h can exceed the fp16 range on Q4_K layers), the
//            shared rows -> bf16; -> hb, hscale
//   down     per (group, 128-row tile of D, chunk): D = Dn_tile . hb_rows^T,
//            epilogue y[slot] = w[slot] * 2^e[slot] * D (fp32; weight 1 and
//            no scale for the shared rows)
//   combine  out[t] = y[6T + t] + sum_{k=0..5} y[inv[t][k]]   (fixed order)
//
// Groups are the 256 routed experts plus the shared expert (group 256).  A
// GEMM CTA is persistent (one per SM) and warp-specialised:
//   warp 0      TMA producer: bucket rows of xb/hb (16-row boxes) and, for the
//               shared expert, its bf16 weight tiles
//   warp 1      TMEM owner and MMA issuer (tcgen05.mma, M = 128, N <= 128)
//   warps 2-5   epilogue (TMEM -> registers -> global)
//   warps 6-21  dequantisers: packed IQ2_XXS / Q2_K / Q4_K tile-blocks are
//               read straight from HBM into registers (one block column
//               prefetched ahead) and written as bf16 into the 128-byte
//               swizzled shared-memory layout the tensor core reads.
// The routed weights enter as the fp32 value of the block formula rounded to
// nearest even in fp16, against fp16 activations (gate/up) and fp16 scaled h
// (down), so the GEMM's only departures from fp32 are that operand rounding
// and the accumulation order.  The shared expert is bf16 throughout (its
// weights are bf16 in memory).
//
// Dequantisation without per-weight arithmetic: an IQ2_XXS sub-block has
// only three magnitudes db*8, db*25, db*43 (the codebook's values), a Q2_K
// sub-block four values d*sc*q - dmin*m.  They are computed once per
// sub-block in fp32, rounded to bf16 and split into a low-byte and a
// high-byte register; each pair of weights is then one byte permute (prmt)
// whose selector comes from a small table indexed by the codes, and, for
// IQ2_XXS, one xor with the pair's sign bits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "ds4g_internal.cuh"
#include "tc.cuh"

namespace ds4g {

constexpr int kBM = 128;        // weight rows per task (MMA M)
constexpr int kBK = 64;         // K per pipeline stage (one 128-byte bf16 row)
constexpr int kNC = 128;        // bucket rows per task (MMA N <= 128)
constexpr int kStages = 3;
constexpr int kTile = kBM * kBK * 2;   // 16 KB: A tile, and the largest B tile
constexpr int kStageBytes = 3 * kTile; // A0, A1, B
constexpr int kDqWarps = 16;   // two threads per weight row and matrix: each takes half of a stage's columns
constexpr int kPFThreads = (6 + kDqWarps) * 32;
constexpr int kGroups = kE + 1;        // routed experts + shared expert

struct PFArgs {
    int T;
    int phase;         // 1 = gate/up, 2 = down
    int qt;            // routed A type
    int hb_q2perm;     // phase 1: store routed h in the Q2_K K-order
    int Mdim, Kdim;
    const int32_t *offsets;          // [257]
    const uint8_t *const *A0;        // phase 1: gate[256]; phase 2: down[256]
    const uint8_t *const *A1;        // phase 1: up[256]
    const uint64_t *grid;
    const int32_t *perm;             // [6T]
    const float *w;                  // [T*6]
    float *h32;                      // [7T][2048] h in fp32 (gate/up output; aliases y)
    const float *hscale;             // [7T] 2^e of each row of hb (down phase)
    float *y;                        // [7T][4096]
    uint32_t *status;
};

// ------------------------------------------------------------ shared memory
struct PFSmem {
    uint8_t *stage;        // kStages x {A0, A1, B}
    uint4 *sel;            // [256][8] IQ2 grid row -> 4 prmt selectors (8 replicas: no bank conflicts)
    uint4 *sgn;            // [128][8] IQ2 sign index -> 4 sign masks
    uint2 *q2lut;          // [256][16] byte of four 2-bit codes -> 2 selectors (phase 2; aliases sel)
    int *tp;               // [258] task prefix over groups
    uint64_t *full_a, *full_b, *empty, *acc_full, *acc_empty;
    uint32_t *tmem_base;
    int *abort_flag;
    uint64_t *drain;       // the MMA thread's final commit: all its MMAs complete
};

constexpr size_t kSmemTables = 256 * 8 * 16 + 128 * 8 * 16 + 1040;   // 48 KB of tables + task prefix
constexpr size_t kSmemBars = (3 * kStages + 4) * 8 + 16;
constexpr size_t kPFSmemBytes = 1024 + (size_t)kStages * kStageBytes + kSmemTables + kSmemBars;

__device__ __forceinline__ PFSmem carve(uint8_t *raw) {
    PFSmem s;
    uint8_t *p = (uint8_t *)(((uintptr_t)raw + 1023) & ~(uintptr_t)1023);
    s.stage = p;
    p += (size_t)kStages * kStageBytes;
    s.sel = (uint4 *)p;
    s.q2lut = (uint2 *)p;
    p += 256 * 8 * 16;
    s.sgn = (uint4 *)p;
    p += 128 * 8 * 16;
    s.tp = (int *)p;
    p += 1040;
    uint64_t *b = (uint64_t *)p;
    s.full_a = b;
    s.full_b = b + kStages;
    s.empty = b + 2 * kStages;
    s.acc_full = b + 3 * kStages;
    s.acc_empty = b + 3 * kStages + 2;
    p += (3 * kStages + 4) * 8;
    s.tmem_base = (uint32_t *)p;
    s.abort_flag = (int *)(p + 4);
    s.drain = (uint64_t *)(p + 8);
    return s;
}

// -------------------------------------------------------------- task list
struct PFTask {
    int g, mt, row0, n, npad;
    bool shared;
};

__device__ __forceinline__ int group_rows(const PFArgs &a, int g) {
    if (g == kE) return a.T;
    const int n = a.offsets[g + 1] - a.offsets[g];
    return n > 0 ? n : 0;
}

__device__ __forceinline__ PFTask decode_task(const PFArgs &a, const int *tp, int tau) {
    int lo = 0, hi = kGroups;  // tp[lo] <= tau < tp[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tp[mid] <= tau) lo = mid;
        else hi = mid;
    }
    const int mtiles = a.Mdim / kBM;
    const int r = tau - tp[lo];
    const int c = r / mtiles;
    PFTask t;
    t.g = lo;
    t.mt = r - c * mtiles;
    t.shared = lo == kE;
    const int base = t.shared ? kK * a.T : a.offsets[lo];
    const int ng = group_rows(a, lo);
    t.row0 = base + c * kNC;
    t.n = min(kNC, ng - c * kNC);
    t.npad = (t.n + 15) & ~15;
    return t;
}

// ------------------------------------------------------------ bounded wait
__device__ __noinline__ bool pf_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (tc::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > (4ll << 30)) return false;  // ~2 s at 2 GHz
    }
}
// The same wait with its first test inline, for the single-thread producer
// and MMA issuer, whose barriers are often complete already.
__device__ __forceinline__ bool pf_wait_fast(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    return tc::mbar_try_wait(bar, parity) || pf_wait(bar, parity, abort_flag);
}

// Bounded wait for one barrier phase at teardown.  It ignores the abort
// flag: a TMA load or an MMA still in flight must finish before the CTA
// releases its shared memory and TMEM.  Gives up after ~2 s (DS4G_ETIMEOUT).
__device__ __forceinline__ void pf_drain(const PFArgs &a, uint64_t *bar, uint32_t parity, uint32_t where) {
    const long long t0 = clock64();
    while (!tc::mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > (4ll << 30)) {
            flag_status(a.status, DS4G_ETIMEOUT, where);
            return;
        }
    }
}

__device__ __forceinline__ void pf_abort(const PFArgs &a, int *abort_flag, uint32_t where) {
    atomicExch(abort_flag, 1);
    flag_status(a.status, DS4G_ETIMEOUT, where);
}

// ---------------------------------------------------------- bf16 helpers
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// Operand element of the GEMM: fp16 for the routed experts (activations are
// RMS-normalised, |x| <= 64, h enters scaled per row, and fp16 keeps 3 more
// bits than bf16), bf16 for the shared expert's activations (its weights are
// bf16 in memory, and both operands of one MMA have the same type).
__device__ __forceinline__ uint32_t pack2(bool f16, float lo, float hi) {
    return f16 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
}
// Byte-split value registers of four 16-bit values v0..v3: lo bytes and hi bytes.
__device__ __forceinline__ void split4(bool f16, float v0, float v1, float v2, float v3, uint32_t &rlo,
                                       uint32_t &rhi) {
    const uint32_t p0 = pack2(f16, v0, v1), p1 = pack2(f16, v2, v3);
    rlo = prmt(p0, p1, 0x6420);
    rhi = prmt(p0, p1, 0x7531);
}
__device__ __forceinline__ float f16lo(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v & 0xffffu))); }
__device__ __forceinline__ float f16hi(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v >> 16))); }

__device__ __forceinline__ uint4 ldg_nc128(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ uint32_t ldg_nc32(const void *p) {
    uint32_t r;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}
__device__ __forceinline__ uint2 ldg_nc64(const void *p) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

__device__ __forceinline__ void sts128(uint8_t *tile, int m, int chunk, uint4 v) {
    *reinterpret_cast<uint4 *>(tile + m * 128 + ((chunk ^ (m & 7)) << 4)) = v;
}

// One dequantiser thread's packed data for one 256-column block column: the
// half of its row segment that its parity `par` of the stage's columns needs.
//   IQ2_XXS (phase 1): the 8-byte records j = 2 ks + par (ks = 0..3): the
//     row's 16-byte words par and 2 + par;
//   Q4_K: the 32-column sub-blocks j = 2 ks + h (h = par in phase 1, the
//     k-half in phase 2): the row's 16-byte words 2h, 2h + 1, 4 + 2h, 5 + 2h,
//     plus the 12 scale bytes;
//   Q2_K (phase 2): the 32-bit words par * 4 .. + 3 of the row's k-half and
//     their scale word.
// The kernel is instantiated per weight type QT, so each instance holds only
// its own type's registers.
template <int QT>
struct BlockRegs {
    uint4 q[QT == DS4G_Q4_K ? 4 : QT == DS4G_IQ2_XXS ? 2 : 1];
    uint32_t s[QT == DS4G_Q4_K ? 3 : 1];
    uint32_t dd;
};

template <int QT>
__device__ __forceinline__ void load_block(const PFArgs &a, const uint8_t *mat, int r, int kb, int kh, int par,
                                           BlockRegs<QT> &R) {
    const int nbc = a.Kdim / 256;
    const int rr = r & 15, g8 = rr & 7, hrow = rr >> 3;
    if constexpr (QT == DS4G_IQ2_XXS) {
        const uint8_t *tb = mat + ((size_t)(r >> 4) * nbc + kb) * kTB_IQ2;
        const uint8_t *row = tb + 512 * hrow + 64 * g8;
        R.q[0] = ldg_nc128(row + 16 * par);
        R.q[1] = ldg_nc128(row + 16 * (2 + par));
        R.dd = ldg_nc32(tb + 1024 + 4 * g8) >> (16 * hrow);
    } else if constexpr (QT == DS4G_Q2_K) {
        const uint8_t *tb = mat + ((size_t)(r >> 4) * nbc + kb) * kTB_Q2K;
        const uint8_t *row = tb + 512 * hrow + 64 * g8 + 32 * kh;
        R.q[0] = ldg_nc128(row + 16 * par);
        R.s[0] = ldg_nc32(tb + 1024 + 128 * hrow + 16 * g8 + 8 * kh + 4 * par);
        R.dd = ldg_nc32(tb + 1280 + 8 * g8 + 4 * hrow);
    } else {  // Q4_K
        const int h = a.phase == 1 ? par : kh;
        const uint8_t *tb = mat + ((size_t)(r >> 4) * nbc + kb) * kTB_Q4K;
        const uint8_t *row = tb + 1024 * hrow + 128 * g8;
        R.q[0] = ldg_nc128(row + 16 * (2 * h));
        R.q[1] = ldg_nc128(row + 16 * (2 * h + 1));
        R.q[2] = ldg_nc128(row + 16 * (4 + 2 * h));
        R.q[3] = ldg_nc128(row + 16 * (5 + 2 * h));
        const uint8_t *sc = tb + 2048 + 12 * rr;
        R.s[0] = ldg_nc32(sc);
        R.s[1] = ldg_nc32(sc + 4);
        R.s[2] = ldg_nc32(sc + 8);
        R.dd = ldg_nc32(tb + 2240 + 8 * g8 + 4 * hrow);
    }
}

// Ask L2 to fetch the packed row segment this thread will need two block
// columns from now (hides HBM latency behind the register double buffer).
template <int QT>
__device__ __forceinline__ void prefetch_block(const PFArgs &a, const uint8_t *mat, int r, int kb, int kh) {
    const int nbc = a.Kdim / 256;
    if (kb >= nbc) return;
    const int rr = r & 15, g8 = rr & 7, hrow = rr >> 3;
    const uint8_t *p;
    if constexpr (QT == DS4G_IQ2_XXS) p = mat + ((size_t)(r >> 4) * nbc + kb) * kTB_IQ2 + 512 * hrow + 64 * g8;
    else if constexpr (QT == DS4G_Q2_K)
        p = mat + ((size_t)(r >> 4) * nbc + kb) * kTB_Q2K + 512 * hrow + 64 * g8 + 32 * kh;
    else p = mat + ((size_t)(r >> 4) * nbc + kb) * kTB_Q4K + 1024 * hrow + 128 * g8;
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

template <int QT>
__device__ __forceinline__ uint32_t word_of(const BlockRegs<QT> &R, int i) {
    const uint4 v = R.q[i >> 2];
    const int k = i & 3;
    return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}
__device__ __forceinline__ uint32_t word4(uint4 v, int k) { return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w; }

// IQ2_XXS: the 32 weights of record j (8 bytes of the row; qw = the 16-byte
// word of the row that holds it) as 4 chunks of 8 fp16 values.  It reads only
// the lookup tables, so the dequantisers build a stage's chunks before they
// wait for the stage to be free, and only store them after.
__device__ __forceinline__ void dq_iq2_record(const PFSmem &sm, const BlockRegs<DS4G_IQ2_XXS> &R, uint4 qw, int j,
                                              int rep8, uint4 (&o)[4]) {
    // record j sits in the row's 16-byte word j & 3, 32-bit words 2 (j >> 2), +1;
    // qw is that 16-byte word
    const uint32_t ia = word4(qw, 2 * (j >> 2)), v = word4(qw, 2 * (j >> 2) + 1);
    const float d = f16lo(R.dd);
    const float db = __fmul_rn(__fmul_rn(d, __fadd_rn(0.5f, (float)(v >> 28))), 0.25f);
    uint32_t rlo, rhi;
    split4(true, __fmul_rn(db, 8.0f), __fmul_rn(db, 25.0f), __fmul_rn(db, 43.0f), 0.0f, rlo, rhi);
#pragma unroll
    for (int l = 0; l < 4; ++l) {
        const uint4 sel = sm.sel[8 * ((ia >> (8 * l)) & 255u) + rep8];
        const uint4 sg = sm.sgn[8 * ((v >> (7 * l)) & 127u) + rep8];
        o[l].x = prmt(rlo, rhi, sel.x) ^ sg.x;
        o[l].y = prmt(rlo, rhi, sel.y) ^ sg.y;
        o[l].z = prmt(rlo, rhi, sel.z) ^ sg.z;
        o[l].w = prmt(rlo, rhi, sel.w) ^ sg.w;
    }
}

// Q2_K: 16 weights of one sub-block (word W, scale byte scb) as 2 chunks (o[0],
// o[1]) in the K-order (0,2,4,...,14,1,3,...,15); like the IQ2_XXS records,
// built before the stage wait and stored after it.
__device__ __forceinline__ void dq_q2k_sub(const PFSmem &sm, uint32_t W, uint32_t scb, float d, float dmin,
                                           int rep16, uint4 (&o)[4]) {
    const float dsc = __fmul_rn(d, (float)(scb & 15u));
    const float dm = __fmul_rn(dmin, (float)(scb >> 4));
    uint32_t rlo, rhi;
    split4(true, __fmaf_rn(dsc, 0.0f, -dm), __fmaf_rn(dsc, 1.0f, -dm), __fmaf_rn(dsc, 2.0f, -dm),
           __fmaf_rn(dsc, 3.0f, -dm), rlo, rhi);
    const uint2 s0 = sm.q2lut[16 * (W & 255u) + rep16], s1 = sm.q2lut[16 * ((W >> 8) & 255u) + rep16];
    const uint2 s2 = sm.q2lut[16 * ((W >> 16) & 255u) + rep16], s3 = sm.q2lut[16 * (W >> 24) + rep16];
    o[0] = make_uint4(prmt(rlo, rhi, s0.x), prmt(rlo, rhi, s0.y), prmt(rlo, rhi, s1.x), prmt(rlo, rhi, s1.y));
    o[1] = make_uint4(prmt(rlo, rhi, s2.x), prmt(rlo, rhi, s2.y), prmt(rlo, rhi, s3.x), prmt(rlo, rhi, s3.y));
}

// Q4_K: weights of sub-block j, 8-column chunks cq0 .. cq0 + ncq - 1 of its 4
// (natural order) -> tile chunks chunk0 + cq, fp32 formula.
__device__ __forceinline__ void dq_q4k_sub(bool f16, const BlockRegs<DS4G_Q4_K> &R, int j, uint4 qv, uint8_t *tile,
                                           int m,
                                           int chunk0, int cq0 = 0, int ncq = 4) {
    const uint32_t s0 = (R.s[0] >> (8 * (j & 3))) & 0xffu;
    const uint32_t s1 = (R.s[1] >> (8 * (j & 3))) & 0xffu;
    const uint32_t s2 = (R.s[2] >> (8 * (j & 3))) & 0xffu;
    uint32_t sc, mn;
    if (j < 4) {
        sc = s0 & 63u;
        mn = s1 & 63u;
    } else {
        sc = (s2 & 15u) | ((s0 >> 6) << 4);
        mn = (s2 >> 4) | ((s1 >> 6) << 4);
    }
    const float dsc = __fmul_rn(f16lo(R.dd), (float)sc);
    const float dm = __fmul_rn(f16hi(R.dd), (float)mn);
    const uint32_t words[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
    for (int cq = 0; cq < 4; ++cq) {  // chunk cq = columns 8cq .. 8cq+7 = c in {2cq, 2cq+1}
        if (cq < cq0 || cq >= cq0 + ncq) continue;
        uint32_t o[4];
#pragma unroll
        for (int pr = 0; pr < 4; ++pr) {  // pair pr: columns 8cq + 2pr, +1
            const int c = 2 * cq + (pr >> 1), p = 2 * (pr & 1);
            const uint32_t x = (words[c >> 1] >> (4 * (2 * (c & 1) + (p >> 1)))) & 0x000F000Fu;
            o[pr] = pack2(f16, __fmaf_rn(dsc, (float)(x & 15u), -dm), __fmaf_rn(dsc, (float)(x >> 16), -dm));
        }
        sts128(tile, m, chunk0 + cq, make_uint4(o[0], o[1], o[2], o[3]));
    }
}

// ------------------------------------------------------------------ kernel
template <int QT>
__global__ void __launch_bounds__(kPFThreads, 1)
    prefill_gemm_kernel(const __grid_constant__ CUtensorMap tmB16, const __grid_constant__ CUtensorMap tmB32,
                        const __grid_constant__ CUtensorMap tmB64, const __grid_constant__ CUtensorMap tmB128,
                        const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1, PFArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const PFSmem sm = carve(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int mtiles = a.Mdim / kBM;
    const int nkb = a.Kdim / kBK;           // stages per task
    const int nmat = a.phase == 1 ? 2 : 1;
    const uint32_t tmem_cols = a.phase == 1 ? 512u : 256u;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(&sm.full_a[s], kDqWarps);
            tc::mbar_init(&sm.full_b[s], 1);
            tc::mbar_init(&sm.empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&sm.acc_full[i], 1);
            tc::mbar_init(&sm.acc_empty[i], 4);
        }
        tc::mbar_init(sm.drain, 1);
        *sm.abort_flag = 0;
        tc::fence_mbar_init();
        tc::prefetch_tmap(&tmB16);
        tc::prefetch_tmap(&tmB32);
        tc::prefetch_tmap(&tmB64);
        tc::prefetch_tmap(&tmB128);
        tc::prefetch_tmap(&tmA0);
        tc::prefetch_tmap(&tmA1);
    }
    if (warp == 1) {
        tc::tmem_alloc(sm.tmem_base, tmem_cols);
        tc::tmem_relinquish();
    }
    // lookup tables of the dequantisers
    if constexpr (QT == DS4G_IQ2_XXS) {
        for (int i = tid; i < 256; i += kPFThreads) {
            const uint64_t row = a.grid[i];
            uint32_t sel[4];
            bool bad = false;
#pragma unroll
            for (int wv = 0; wv < 4; ++wv) {
                uint32_t lv[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t g = (uint32_t)(row >> (8 * (2 * wv + h))) & 255u;
                    lv[h] = g == 8 ? 0u : g == 25 ? 1u : g == 43 ? 2u : 3u;
                    bad |= lv[h] == 3u;
                }
                sel[wv] = lv[0] | ((lv[0] + 4) << 4) | (lv[1] << 8) | ((lv[1] + 4) << 12);
            }
            if (bad) flag_status(a.status, DS4G_EUNSUPPORTED, 0x6D1Du);
            const uint4 v4 = make_uint4(sel[0], sel[1], sel[2], sel[3]);
#pragma unroll
            for (int r = 0; r < 8; ++r) sm.sel[8 * i + r] = v4;
        }
        for (int i = tid; i < 128; i += kPFThreads) {
            const uint32_t s = (uint32_t)i | ((uint32_t)(__popc(i) & 1) << 7);
            uint32_t mk[4];
#pragma unroll
            for (int wv = 0; wv < 4; ++wv)
                mk[wv] = (((s >> (2 * wv)) & 1u) << 15) | (((s >> (2 * wv + 1)) & 1u) << 31);
            const uint4 v4 = make_uint4(mk[0], mk[1], mk[2], mk[3]);
#pragma unroll
            for (int r = 0; r < 8; ++r) sm.sgn[8 * i + r] = v4;
        }
    }
    if constexpr (QT == DS4G_Q2_K) {
        for (int x = tid; x < 256; x += kPFThreads) {
            uint32_t sel[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t c0 = (x >> (4 * h)) & 3u, c1 = (x >> (4 * h + 2)) & 3u;
                sel[h] = c0 | ((c0 + 4) << 4) | (c1 << 8) | ((c1 + 4) << 12);
            }
            const uint2 v2 = make_uint2(sel[0], sel[1]);
#pragma unroll
            for (int r = 0; r < 16; ++r) sm.q2lut[16 * x + r] = v2;
        }
    }
    // task prefix over the groups (warp 2; 9 groups per lane)
    if (warp == 2) {
        int cnt[9], s = 0;
#pragma unroll
        for (int i = 0; i < 9; ++i) {
            const int g = lane * 9 + i;
            int c = 0;
            if (g < kGroups) c = (group_rows(a, g) + kNC - 1) / kNC * mtiles;
            cnt[i] = c;
            s += c;
        }
        int inc = s;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += o;
        }
        int run = inc - s;
#pragma unroll
        for (int i = 0; i < 9; ++i) {
            const int g = lane * 9 + i;
            run += cnt[i];
            if (g < kGroups) sm.tp[g + 1] = run;
        }
        if (lane == 0) sm.tp[0] = 0;
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tbase = *sm.tmem_base;
    const int ntask = sm.tp[kGroups];
    volatile int *abort_flag = sm.abort_flag;

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0) {
            uint32_t it = 0, pph = 0;
            int ps = 0;
            for (int tau = blockIdx.x; tau < ntask && !*abort_flag; tau += gridDim.x) {
                const PFTask t = decode_task(a, sm.tp, tau);
                // one box per stage: the smallest of 16/32/64/128 rows covering the chunk
                const int brows = t.npad <= 16 ? 16 : t.npad <= 32 ? 32 : t.npad <= 64 ? 64 : 128;
                const CUtensorMap *tmB = brows == 16 ? &tmB16 : brows == 32 ? &tmB32 : brows == 64 ? &tmB64 : &tmB128;
                const uint32_t bytes = (uint32_t)brows * 128u + (t.shared ? (uint32_t)nmat * kTile : 0u);
                for (int ks = 0; ks < nkb; ++ks, ++it) {
                    const int s = ps;
                    const uint32_t ph = pph;
                    if (++ps == kStages) {   // stage and phase of the next load
                        ps = 0;
                        pph ^= 1u;
                    }
                    if (!pf_wait_fast(&sm.empty[s], ph ^ 1u, abort_flag)) {
                        pf_abort(a, sm.abort_flag, 0x100u);
                        break;
                    }
                    uint8_t *st = sm.stage + (size_t)s * kStageBytes;
                    tc::mbar_arrive_expect_tx(&sm.full_b[s], bytes);
                    tc::tma_load_2d(st + 2 * kTile, tmB, ks * kBK, t.row0, &sm.full_b[s]);
                    if (t.shared) {
                        tc::tma_load_2d(st, &tmA0, ks * kBK, t.mt * kBM, &sm.full_b[s]);
                        if (nmat == 2) tc::tma_load_2d(st + kTile, &tmA1, ks * kBK, t.mt * kBM, &sm.full_b[s]);
                    }
                }
            }
            // the last load issued into each stage has landed (already so when
            // the MMA thread consumed everything; after an abort this keeps
            // loads from writing shared memory after exit)
            for (uint32_t u = 0; u < (uint32_t)kStages; ++u) {
                if (it <= u) continue;   // stage never used
                const uint32_t last = it - 1 - (it - 1 - u) % kStages;
                pf_drain(a, &sm.full_b[u], (last / kStages) & 1u, 0x500u + u);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            uint32_t ti = 0, ph = 0;   // stage s and phase ph of the next stage
            int s = 0;
            for (int tau = blockIdx.x; tau < ntask && !*abort_flag; tau += gridDim.x, ++ti) {
                const PFTask t = decode_task(a, sm.tp, tau);
                const int ab = ti & 1;
                if (!pf_wait(&sm.acc_empty[ab], ((ti >> 1) & 1u) ^ 1u, abort_flag)) {
                    pf_abort(a, sm.abort_flag, 0x200u);
                    break;
                }
                tc::tc_fence_after();
                // routed experts: fp16 operands; shared expert: bf16
                const uint32_t idesc = tc::idesc_f16(kBM, t.npad, t.shared);
                const uint32_t dcol = tbase + (uint32_t)(ab * (a.phase == 1 ? 256 : 128));
                bool ok = true;
                for (int ks = 0; ks < nkb; ++ks) {
                    if (!pf_wait_fast(&sm.full_b[s], ph, abort_flag) || !pf_wait_fast(&sm.full_a[s], ph, abort_flag)) {
                        pf_abort(a, sm.abort_flag, 0x201u);
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    // the A1 and B tiles follow A0 at kTile and 2 kTile bytes (the
                    // descriptors' start-address field counts 16-byte units)
                    const uint64_t da0 = tc::sw128_desc(tc::smem_u32(sm.stage + (size_t)s * kStageBytes));
                    const uint64_t da1 = da0 + (kTile >> 4), db = da0 + (2 * kTile >> 4);
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        const uint32_t acc = (ks > 0 || k4 > 0) ? 1u : 0u;
                        tc::mma_f16_ss(dcol, da0 + 2 * k4, db + 2 * k4, idesc, acc);
                    }
                    if (nmat == 2) {
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4) {
                            const uint32_t acc = (ks > 0 || k4 > 0) ? 1u : 0u;
                            tc::mma_f16_ss(dcol + 128, da1 + 2 * k4, db + 2 * k4, idesc, acc);
                        }
                    }
                    tc::mma_commit(&sm.empty[s]);
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                tc::mma_commit(&sm.acc_full[ab]);
            }
            // every MMA issued here has completed before TMEM is released
            tc::mma_commit(sm.drain);
            pf_drain(a, sm.drain, 0, 0x600u);
        }
    } else if (warp < 6) {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quarter of this warp
        const int m = 32 * q + lane;
        uint32_t ti = 0;
        for (int tau = blockIdx.x; tau < ntask && !*abort_flag; tau += gridDim.x, ++ti) {
            const PFTask t = decode_task(a, sm.tp, tau);
            const int ab = ti & 1;
            if (!pf_wait(&sm.acc_full[ab], (ti >> 1) & 1u, abort_flag)) {
                pf_abort(a, sm.abort_flag, 0x300u);
                break;
            }
            tc::tc_fence_after();
            const int row = t.mt * kBM + m;  // output feature of this lane
            const uint32_t lane_base = tbase + ((uint32_t)(32 * q) << 16);
            if (a.phase == 1) {
                int pos = row;
                if (!t.shared && a.hb_q2perm) pos = (row & ~15) | ((row & 1) << 3) | ((row & 15) >> 1);
                const uint32_t cg = lane_base + (uint32_t)(ab * 256);
                for (int c0 = 0; c0 < t.npad; c0 += 16) {
                    uint32_t g[16], u[16];
                    tc::tmem_ld16(cg + c0, g);
                    tc::tmem_ld16(cg + 128 + c0, u);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int n = c0 + j;
                        if (n < t.n) {
                            const float gv = __uint_as_float(g[j]), uv = __uint_as_float(u[j]);
                            a.h32[(size_t)(t.row0 + n) * kF + pos] = silu_f(gv) * uv;
                        }
                    }
                }
            } else {
                const uint32_t cd = lane_base + (uint32_t)(ab * 128);
                for (int c0 = 0; c0 < t.npad; c0 += 16) {
                    uint32_t dv[16];
                    tc::tmem_ld16(cd + c0, dv);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int n = c0 + j;
                        if (n < t.n) {
                            const int slot = t.row0 + n;
                            const float sc = t.shared ? 1.0f : __ldg(a.w + a.perm[slot]) * __ldg(a.hscale + slot);
                            a.y[(size_t)slot * kH + row] = sc * __uint_as_float(dv[j]);
                        }
                    }
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&sm.acc_empty[ab]);
        }
    } else {
        // ---------------------------------------------------- dequantisers
        const int dq = tid - 6 * 32;           // 0..511
        const int m = dq & 127;
        const int half = (dq >> 7) & 1;        // phase 1: matrix; phase 2: k-half
        const int par = dq >> 8;               // which half of the stage's work of (m, half)
        const int nblk = a.Kdim / 256;
        uint32_t it = 0;
        BlockRegs<QT> cur, nxt;
        // first block of the first task
        int tau = blockIdx.x;
        PFTask t;
        if (tau < ntask) {
            t = decode_task(a, sm.tp, tau);
            if (!t.shared) {
                const uint8_t *mat = (a.phase == 1 && half) ? a.A1[t.g] : a.A0[t.g];
                load_block(a, mat, t.mt * kBM + m, 0, half, par, cur);
            }
        }
        for (; tau < ntask && !*abort_flag; tau += gridDim.x) {
            const uint8_t *mat = nullptr;
            if (!t.shared) mat = (a.phase == 1 && half) ? a.A1[t.g] : a.A0[t.g];
            const int r = t.mt * kBM + m;
            PFTask tn;
            const int taun = tau + gridDim.x;
            if (taun < ntask) tn = decode_task(a, sm.tp, taun);
            bool ok = true;
            for (int kb = 0; kb < nblk && ok; ++kb) {
                // prefetch the next block column (possibly of the next task)
                if (kb + 1 < nblk) {
                    if (!t.shared) {
                        load_block(a, mat, r, kb + 1, half, par, nxt);
                        prefetch_block<QT>(a, mat, r, kb + 2, half);
                    }
                } else if (taun < ntask && !tn.shared) {
                    const uint8_t *matn = (a.phase == 1 && half) ? a.A1[tn.g] : a.A0[tn.g];
                    load_block(a, matn, tn.mt * kBM + m, 0, half, par, nxt);
                }
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const int s = (it + ks) % kStages;
                    const uint32_t ph = ((it + ks) / kStages) & 1u;
                    if (!ok) continue;
                    uint4 o[4];   // IQ2_XXS / Q2_K: this stage's chunks, built before the wait
                    if constexpr (QT == DS4G_IQ2_XXS) {
                        // record 2 ks + par: the row's 16-byte word 2 (ks & 1) + par, held as cur.q[ks & 1]
                        if (!t.shared) dq_iq2_record(sm, cur, cur.q[ks & 1], 2 * ks + par, lane & 7, o);
                    } else if constexpr (QT == DS4G_Q2_K) {
                        // word ks of this thread's 4 (row word 4 par + ks)
                        if (!t.shared)
                            dq_q2k_sub(sm, word_of(cur, ks), (cur.s[0] >> (8 * ks)) & 255u, f16lo(cur.dd),
                                       f16hi(cur.dd), lane & 15, o);
                    }
                    if (!pf_wait_fast(&sm.empty[s], ph ^ 1u, abort_flag)) {
                        pf_abort(a, sm.abort_flag, 0x400u);
                        ok = false;
                        continue;
                    }
                    if (!t.shared) {
                        uint8_t *st = sm.stage + (size_t)s * kStageBytes;
                        if (a.phase == 1) {
                            uint8_t *tile = st + half * kTile;
                            // record / sub-block 2 ks + par -> chunks 4 par .. 4 par + 3
                            if constexpr (QT == DS4G_IQ2_XXS) {
#pragma unroll
                                for (int l = 0; l < 4; ++l) sts128(tile, m, 4 * par + l, o[l]);
                            } else if constexpr (QT == DS4G_Q4_K) {
                                // sub-block j = row word 2 (j & 3) + (j >> 2), held as cur.q[2 (ks & 1) + (ks >> 1)]
                                const int j = 2 * ks + par;
                                dq_q4k_sub(true, cur, j, cur.q[2 * (ks & 1) + (ks >> 1)], tile, m, 4 * par);
                            }
                        } else {
                            if constexpr (QT == DS4G_Q2_K) {
                                // -> chunks 4 half + 2 par, + 1
                                sts128(st, m, 4 * half + 2 * par, o[0]);
                                sts128(st, m, 4 * half + 2 * par + 1, o[1]);
                            } else if constexpr (QT == DS4G_Q4_K) {
                                // sub-block j = 2 ks + half, chunks 2 par, 2 par + 1 of its 4
                                const int j = 2 * ks + half;
                                dq_q4k_sub(true, cur, j, cur.q[2 * (ks & 1) + (ks >> 1)], st, m, 4 * half, 2 * par,
                                           2);
                            }
                        }
                        tc::fence_proxy_async_smem();
                    }
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&sm.full_a[s]);
                }
                it += 4;
                cur = nxt;
            }
            if (!ok) break;
            t = tn;
        }
    }

    // ------------------------------------------------------------ teardown
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tbase, tmem_cols);
    }
}

// ----------------------------------------------------------- permute / cast
// Row r < n_routed: fp16 of the hidden row of the token owning slot perm[r];
// rows n_routed..6T-1 (entries with a bad id) are zero; row 6T + t: bf16 of
// token t (the shared expert's operand).  |x| >= 65504 is flagged.
__global__ void __launch_bounds__(256) permute_cast_kernel(const float *__restrict__ x, const int32_t *perm,
                                                           const int32_t *offsets, int T,
                                                           __nv_bfloat16 *__restrict__ xb, uint32_t *status) {
    const int r = blockIdx.x;
    const int nrt = kK * T;
    int src = -1;
    if (r < nrt) {
        if (r < offsets[kE]) src = perm[r] / kK;
    } else {
        src = r - nrt;
    }
    uint4 *dst = reinterpret_cast<uint4 *>(xb + (size_t)r * kH) + 2 * threadIdx.x;
    if (src < 0) {
        dst[0] = make_uint4(0, 0, 0, 0);
        dst[1] = make_uint4(0, 0, 0, 0);
        return;
    }
    const bool f16 = r < nrt;
    const float4 *xs = reinterpret_cast<const float4 *>(x + (size_t)src * kH) + 4 * threadIdx.x;
    uint32_t o[8];
    bool big = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 v = xs[i];
        big |= !(fabsf(v.x) < 65504.f) || !(fabsf(v.y) < 65504.f) || !(fabsf(v.z) < 65504.f) ||
               !(fabsf(v.w) < 65504.f);
        o[2 * i] = pack2(f16, v.x, v.y);
        o[2 * i + 1] = pack2(f16, v.z, v.w);
    }
    if (big && f16) flag_status(status, DS4G_EDEVICE, 0xF16u);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// Row r of h32 (2048 fp32 values, one CTA of 256 threads): routed rows
// (r < 6T) -> hb = fp16 of 2^-e h, where 2^e puts the row's largest |h| in
// [2^14, 2^15) (any finite h fits fp16 and keeps 11 significant bits), and
// hscale[r] = 2^e; shared rows (r >= 6T) -> bf16 of h, hscale = 1.  The
// routed rows past offsets[256] (entries with a bad id, which no GEMM task
// writes or reads) become zeros.  A non-finite h is flagged.
__global__ void __launch_bounds__(256) hcast_kernel(const float *__restrict__ h32, const int32_t *offsets, int T,
                                                    uint16_t *__restrict__ hb, float *__restrict__ hscale,
                                                    uint32_t *status) {
    const int r = blockIdx.x;
    const bool routed = r < kK * T;
    if (routed && r >= offsets[kE]) {
        *reinterpret_cast<uint4 *>(hb + (size_t)r * kF + 8 * threadIdx.x) = make_uint4(0, 0, 0, 0);
        if (threadIdx.x == 0) hscale[r] = 1.0f;
        return;
    }
    const float4 *src = reinterpret_cast<const float4 *>(h32 + (size_t)r * kF) + 2 * threadIdx.x;
    const float4 v0 = __ldcs(src), v1 = __ldcs(src + 1);
    const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) bad |= !(fabsf(v[i]) <= 3.4028235e38f);
    if (bad) flag_status(status, DS4G_EDEVICE, 0xF16u);
    float e2 = 1.0f;
    if (routed) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        __shared__ float red[8];
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
        __syncthreads();
        m = red[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) m = fmaxf(m, red[i]);
        // m < 2^E with E = biased exponent - 126; e = E - 15 (0 for m = 0)
        const int E = (int)((__float_as_uint(m) >> 23) & 255u) - 126;
        const int e = m > 0.f ? max(min(E - 15, 100), -100) : 0;
        e2 = __uint_as_float((uint32_t)(127 + e) << 23);
        const float inv = __uint_as_float((uint32_t)(127 - e) << 23);
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = pack_f16x2(v[2 * i] * inv, v[2 * i + 1] * inv);
        *reinterpret_cast<uint4 *>(hb + (size_t)r * kF + 8 * threadIdx.x) = make_uint4(o[0], o[1], o[2], o[3]);
    } else {
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
        *reinterpret_cast<uint4 *>(hb + (size_t)r * kF + 8 * threadIdx.x) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (threadIdx.x == 0) hscale[r] = e2;
}

// out[t] = y[6T + t] + sum_{k=0..5} y[inv[6t + k]]   (fixed order)
__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ y, const int32_t *inv, int T,
                                                      float *__restrict__ out) {
    const int t = blockIdx.x;
    int src[kK];
#pragma unroll
    for (int k = 0; k < kK; ++k) src[k] = inv[t * kK + k];
    const float4 *ys = reinterpret_cast<const float4 *>(y + (size_t)(kK * T + t) * kH);
    float4 *o = reinterpret_cast<float4 *>(out + (size_t)t * kH);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int c = threadIdx.x + 256 * i;
        float4 acc = __ldcs(ys + c);
#pragma unroll
        for (int k = 0; k < kK; ++k) {
            if (src[k] < 0) continue;
            const float4 v = __ldcs(reinterpret_cast<const float4 *>(y + (size_t)src[k] * kH) + c);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        o[c] = acc;
    }
}

// ------------------------------------------------------------------- host
struct PFLayout {
    size_t counts, offsets, perm, inv, hscale, xb, hb, y, total;
};

static PFLayout pf_layout(int T) {
    PFLayout L;
    const size_t nslot = (size_t)kK * T, nrow = nslot + T;
    size_t off = kWsScratch;   // the counter area below stays untouched
    L.counts = off;
    off += align_up(kE * 4, 256);
    L.offsets = off;
    off += align_up((kE + 1) * 4, 256);
    L.perm = off;
    off += align_up(nslot * 4, 256);
    L.inv = off;
    off += align_up(nslot * 4, 256);
    L.hscale = off;
    off += align_up(nrow * 4, 256);
    L.xb = off;
    off += align_up(nrow * kH * 2, 1024);
    L.hb = off;
    off += align_up(nrow * kF * 2, 1024);
    L.y = off;
    off += align_up(nrow * kH * 4, 256);
    L.total = off;
    return L;
}

size_t prefill_workspace(int T) { return pf_layout(T).total; }

ds4g_status bucket_launch(const int32_t *ids, int T, int32_t *counts, int32_t *offsets, int32_t *perm,
                          int32_t *inv, uint32_t *status, cudaStream_t st);

static int g_pf_sms = 0;
static bool g_pf_attr = false;

// One instance per weight type: IQ2_XXS (gate/up), Q2_K (down), Q4_K (both).
template <int QT>
static cudaError_t pf_launch_t(const CUtensorMap (&mB)[4], const CUtensorMap &m0, const CUtensorMap &m1,
                               const PFArgs &a, cudaStream_t st) {
    prefill_gemm_kernel<QT><<<g_pf_sms, kPFThreads, kPFSmemBytes, st>>>(mB[0], mB[1], mB[2], mB[3], m0, m1, a);
    return cudaGetLastError();
}
static cudaError_t pf_launch(const CUtensorMap (&mB)[4], const CUtensorMap &m0, const CUtensorMap &m1,
                             const PFArgs &a, cudaStream_t st) {
    switch (a.qt) {
    case DS4G_IQ2_XXS: return pf_launch_t<DS4G_IQ2_XXS>(mB, m0, m1, a, st);
    case DS4G_Q2_K: return pf_launch_t<DS4G_Q2_K>(mB, m0, m1, a, st);
    case DS4G_Q4_K: return pf_launch_t<DS4G_Q4_K>(mB, m0, m1, a, st);
    default: return cudaErrorInvalidValue;
    }
}

// phases: 1 = bucket, permute and gate/up; 2 = down and combine; 3 = both.
ds4g_status prefill_forward(const float *hidden, int T, const ds4g_layer *L, const int32_t *ids, const float *w,
                            float *out, void *workspace, cudaStream_t st, int phases) {
    if (!g_pf_sms) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return DS4G_ECUDA;
        if (cudaDeviceGetAttribute(&g_pf_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return DS4G_ECUDA;
    }
    if (!g_pf_attr) {
        if (cudaFuncSetAttribute(prefill_gemm_kernel<DS4G_IQ2_XXS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kPFSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(prefill_gemm_kernel<DS4G_Q2_K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kPFSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(prefill_gemm_kernel<DS4G_Q4_K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kPFSmemBytes) != cudaSuccess)
            return DS4G_ECUDA;
        g_pf_attr = true;
    }
    uint8_t *ws = (uint8_t *)workspace;
    const PFLayout lay = pf_layout(T);
    uint32_t *status = (uint32_t *)ws;
    int32_t *counts = (int32_t *)(ws + lay.counts), *offsets = (int32_t *)(ws + lay.offsets);
    int32_t *perm = (int32_t *)(ws + lay.perm), *inv = (int32_t *)(ws + lay.inv);
    __nv_bfloat16 *xb = (__nv_bfloat16 *)(ws + lay.xb), *hb = (__nv_bfloat16 *)(ws + lay.hb);
    float *y = (float *)(ws + lay.y);
    float *hscale = (float *)(ws + lay.hscale);
    const int nrow = (kK + 1) * T;

    PFArgs a;
    a.T = T;
    a.offsets = offsets;
    a.grid = L->iq2_grid;
    a.perm = perm;
    a.w = w;
    a.h32 = y;        // gate/up output; consumed by the cast before the down phase writes y
    a.hscale = hscale;
    a.y = y;
    a.status = status;
    if (phases & 1) {
        ds4g_status rc = bucket_launch(ids, T, counts, offsets, perm, inv, status, st);
        if (rc != DS4G_OK) return rc;
        permute_cast_kernel<<<nrow, 256, 0, st>>>(hidden, perm, offsets, T, xb, status);
        if (cudaGetLastError() != cudaSuccess) return DS4G_ECUDA;
        CUtensorMap mB[4], mG, mU;
        for (int i = 0; i < 4; ++i)
            if (!tmap_bf16_2d(&mB[i], xb, nrow, kH, 16u << i)) return DS4G_ECUDA;
        if (!tmap_bf16_2d(&mG, L->sh_gate, kF, kH, kBM) || !tmap_bf16_2d(&mU, L->sh_up, kF, kH, kBM)) return DS4G_ECUDA;
        a.phase = 1;
        a.qt = L->gate_up_type;
        a.hb_q2perm = L->down_type == DS4G_Q2_K ? 1 : 0;
        a.Mdim = kF;
        a.Kdim = kH;
        a.A0 = reinterpret_cast<const uint8_t *const *>(L->gate);
        a.A1 = reinterpret_cast<const uint8_t *const *>(L->up);
        if (pf_launch(mB, mG, mU, a, st) != cudaSuccess) return DS4G_ECUDA;
    }
    if (!(phases & 2)) return DS4G_OK;
    hcast_kernel<<<nrow, 256, 0, st>>>(y, offsets, T, reinterpret_cast<uint16_t *>(hb), hscale, status);
    if (cudaGetLastError() != cudaSuccess) return DS4G_ECUDA;
    CUtensorMap mB2[4], mD;
    for (int i = 0; i < 4; ++i)
        if (!tmap_bf16_2d(&mB2[i], hb, nrow, kF, 16u << i)) return DS4G_ECUDA;
    if (!tmap_bf16_2d(&mD, L->sh_down, kH, kF, kBM)) return DS4G_ECUDA;
    a.phase = 2;
    a.qt = L->down_type;
    a.hb_q2perm = 0;
    a.Mdim = kH;
    a.Kdim = kF;
    a.A0 = reinterpret_cast<const uint8_t *const *>(L->down);
    a.A1 = nullptr;
    if (pf_launch(mB2, mD, mD, a, st) != cudaSuccess) return DS4G_ECUDA;
    combine_kernel<<<T, 256, 0, st>>>(y, inv, T, out);
    if (cudaGetLastError() != cudaSuccess) return DS4G_ECUDA;
    return DS4G_OK;
}

}  // namespace ds4g
