// decode1.cu — one decode token through one MoE layer in a single launch
// (chenxutan ds4 article §2.3: router logic and expert compute fused into one
// GPU dispatch, hard-coded graph; §3.2: router -> only the routed experts'
// weights -> shared expert -> merge).  For T = 1 with IQ2_XXS/Q2_K experts.
//
// One persistent CTA per SM, 18 warps: a producer warp, a router warp and
// four consumer groups of four warps.  Each CTA owns a static list of jobs in
// five phases — router rows, shared gate/up rows, routed gate/up 16-row tiles,
// shared down row pairs, routed down (expert, 16-row tile) — phase p's jobs
// dealt round-robin over the CTAs in alternating direction so per-CTA totals
// balance, and the CTA's jobs dealt round-robin to its groups.  The producer
// streams every weight piece (<= 8.5 KB, contiguous) of a group's jobs into
// the group's four-slot shared-memory ring with cp.async.bulk, so each SM
// keeps up to twelve pieces (~100 KB) in flight.  A group splits each piece
// over its four warps, keeps partials in registers until the job's last
// piece and reduces them in a fixed order behind a four-warp barrier.
//
// Dependencies are exactly those of the method:
//  - expert ids: every CTA's router warp waits until all 256 router logits
//    are stored, then computes the top-6 itself (all CTAs get the same ids);
//    the producer streams routed pieces only after that;
//  - h: a CTA enters the down phase once every CTA has stored its gate/up h
//    (one release per CTA); down weights keep streaming meanwhile;
//  - out: the shared-row jobs and the six routed jobs of a 16-row output tile
//    store partials; the last of the 14 to finish (a per-tile counter) sums
//    them in a fixed order.
// Each CTA waits only for work that running CTAs own, and every wait is
// bounded (~1 s); a timeout records DS4G_ETIMEOUT.
//
// Arithmetic: router and shared expert in fp32 FMA (bf16 weights widen
// exactly); routed experts on mma.sync with exact codes (IQ2 grid value or
// Q2_K quant as an fp16 subnormal, sign from the sign table) against the
// activation as an fp16 hi + lo pair; block and sub-block scales applied in
// fp32 to each 32- or 16-column partial.
#include "ds4g_internal.cuh"
#include "tc.cuh"

namespace ds4g {

constexpr int kNGrp = 4;                         // consumer groups
constexpr int kGW = 4;                           // warps per group
constexpr int kD1Cons = kNGrp * kGW;             // 16 consumer warps
constexpr int kD1Threads = (2 + kD1Cons) * 32;   // producer + router + consumers
constexpr int kD1Slot = 16896;                   // 16 x 1056: an IQ2 row tile, the largest piece
constexpr int kSlotsPerGrp = 2;                  // one piece in flight while one is computed
constexpr int kD1Slots = kNGrp * kSlotsPerGrp;   // 16

// Jobs per phase, in order, and their pieces (each one contiguous copy of
// about 16 KB: a bulk copy has a fixed cost, so pieces are kept large):
//   router rows                       1 piece (16 KB)
//   shared gate/up row pairs          2 pieces (gate rows, up rows: 16 KB each)
//   shared down 4-row groups          1 piece (16 KB)
//   routed gate/up (slot, 16-row tile) 2 pieces (gate, up: 16 tile-blocks each)
//   routed down (slot, 16-row tile)   1 piece (8 Q2_K tile-blocks, 10.5 KB)
constexpr int kNPhase = 5;
constexpr int kJR = kE;
constexpr int kJSG = kF / 2;
constexpr int kJSD = kH / 4;
constexpr int kJRG = kK * (kF / 16);
constexpr int kJRD = kK * (kH / 16);
constexpr int kTileParts = 4 + kK;      // jobs contributing to one 16-row output tile

enum : int { PK_END = 0, PK_ROUTER, PK_SGU, PK_RGU, PK_SDN, PK_RDN };

struct D1Desc {
    int kind, job, piece, e;
};

// Global coordination block (in the workspace; zero before the first launch;
// the last CTA of every launch resets it).
struct D1Sync {
    uint32_t router_done;
    uint32_t sgu_done;     // shared gate/up rows stored
    uint32_t gu_cta;       // CTAs whose routed gate/up jobs are all stored
    uint32_t exit_count;
    uint32_t pad[12];
    uint32_t tile_cnt[kH / 16];
};

struct D1Args {
    const float *x;
    int normalize;
    const float *router;   // [256][4096]
    const float *bias;     // [256]
    int32_t *ids;          // [6] out
    float *w;              // [6] out
    const uint8_t *const *gate;
    const uint8_t *const *up;
    const uint8_t *const *down;
    const __nv_bfloat16 *sh_gate, *sh_up, *sh_down;
    const uint64_t *grid;
    float *out;            // [4096]
    uint32_t *status;
    D1Sync *sync;
    float *logits;         // [256]
    float *h_r;            // [6][2048]
    float *h_s;            // [2048]
    float *p_s;            // [4096] shared-expert output
    float *p_r;            // [6][4096] weighted routed outputs
};

// ------------------------------------------------------------------ smem
// Compile-time offsets from the start of dynamic shared memory.
constexpr uint32_t kOffRing = 0;
constexpr uint32_t kOffDesc = kOffRing + kD1Slots * kD1Slot;
constexpr uint32_t kOffU = kOffDesc + kD1Slots * 16;
constexpr uint32_t kUnion = 256 * 16 * 8 + 128 * 8 * 8 + kH * 4 + 2 * kH * 2;  // 72 KB (phase B uses 52 KB)
constexpr uint32_t kOffHs = kOffU + kUnion;      // shared h (fp32), outside the union
constexpr uint32_t kOffRed = kOffHs + kF * 4;
constexpr uint32_t kOffZero = kOffRed + kNGrp * 2 * 128 * 4;
constexpr uint32_t kOffWk = kOffZero + 512;
constexpr uint32_t kOffIds = kOffWk + 32;
constexpr uint32_t kOffEptr = kOffIds + 32;      // 18 expert matrix pointers (gate, up, down x 6)
constexpr uint32_t kOffCred = kOffEptr + 18 * 8;
constexpr uint32_t kOffBar = kOffCred + 64;
constexpr uint32_t kOffFlags = kOffBar + 2 * kD1Slots * 8;
constexpr size_t kD1SmemBytes = kOffFlags + 16;

struct D1Smem {
    uint8_t *ring;
    D1Desc *desc;
    uint2 *gtab;           // [256][16]   (phase A)
    uint2 *stab;           // [128][8]
    float *xn;             // [4096]
    __half *xq;            // [2][4096] hi, lo
    __half *hq;            // [6][2][2048] (phase B, aliases phase A)
    float *xs16;           // [6][128]
    float *hs;             // [2048] shared h (its own region)
    float *red;            // [4 groups][2][128]
    __half *zero;          // [256] zeros: operand of the inactive mma lanes
    float *wk;             // [6]
    int *ids_s;            // [6]
    const uint8_t **eptr;  // [18] gate[6], up[6], down[6] of the selected experts (NULL if unusable)
    float *cta_red;        // [16]
    uint64_t *full, *empty;
    int *flags;            // [0] abort, [1] ids ready, [2] shared h: 0 absent, 1 loading, 2 present
};

extern __shared__ __align__(1024) uint8_t d1_raw[];

__device__ __forceinline__ D1Smem d1_smem() {
    D1Smem s;
    s.ring = d1_raw + kOffRing;
    s.desc = reinterpret_cast<D1Desc *>(d1_raw + kOffDesc);
    s.gtab = reinterpret_cast<uint2 *>(d1_raw + kOffU);
    s.stab = s.gtab + 256 * 16;
    s.xn = reinterpret_cast<float *>(s.stab + 128 * 8);
    s.xq = reinterpret_cast<__half *>(s.xn + kH);
    s.hq = reinterpret_cast<__half *>(d1_raw + kOffU);
    s.xs16 = reinterpret_cast<float *>(s.hq + kK * 2 * kF);
    s.hs = reinterpret_cast<float *>(d1_raw + kOffHs);
    s.red = reinterpret_cast<float *>(d1_raw + kOffRed);
    s.zero = reinterpret_cast<__half *>(d1_raw + kOffZero);
    s.wk = reinterpret_cast<float *>(d1_raw + kOffWk);
    s.ids_s = reinterpret_cast<int *>(d1_raw + kOffIds);
    s.eptr = reinterpret_cast<const uint8_t **>(d1_raw + kOffEptr);
    s.cta_red = reinterpret_cast<float *>(d1_raw + kOffCred);
    s.full = reinterpret_cast<uint64_t *>(d1_raw + kOffBar);
    s.empty = s.full + kD1Slots;
    s.flags = reinterpret_cast<int *>(d1_raw + kOffFlags);
    return s;
}

// ------------------------------------------------------------- helpers
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     tc::smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Publication with release/acquire ordering (no full fence): a release
// orders this thread's earlier writes, and the writes it has observed through
// a CTA barrier, before the flag or counter update.
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ void red_add_release(uint32_t *p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_release(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded spin until *p >= target.  Returns false on timeout or abort.
__device__ __noinline__ bool spin_geq(const uint32_t *p, uint32_t target, volatile int *abort_flag) {
    const long long t0 = clock64();
    while (true) {
        for (int i = 0; i < 32; ++i)
            if (ld_acquire(p) >= target) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > (2ll << 30)) return false;  // ~1 s
        __nanosleep(64);
    }
}

__device__ __forceinline__ bool d1_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (tc::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > (2ll << 30)) return false;
    }
}

__device__ __forceinline__ void d1_abort(const D1Args &a, int *abort_flag, uint32_t where) {
    atomicExch(abort_flag, 1);
    flag_status(a.status, DS4G_ETIMEOUT, where);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// bf16 x 8 (one uint4) dotted with 8 fp32 values
__device__ __forceinline__ float dot8_bf16(uint4 wv, const float *xv, float acc) {
    const uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc = fmaf(__uint_as_float(wd[i] << 16), xv[2 * i], acc);
        acc = fmaf(__uint_as_float(wd[i] & 0xffff0000u), xv[2 * i + 1], acc);
    }
    return acc;
}

// ------------------------------------------------------ piece consumers
// A router row (4096 fp32) against xn: warp wq takes columns [1024 wq, +1024);
// returns this lane's partial.
__device__ __forceinline__ float router_row(const D1Smem &sm, const uint8_t *slot, int wq, int lane) {
    const float4 *r = reinterpret_cast<const float4 *>(slot) + 256 * wq + lane;
    const float4 *x = reinterpret_cast<const float4 *>(sm.xn) + 256 * wq + lane;
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 rv = r[32 * i], xv = x[32 * i];
        float &acc = (i & 1) ? acc1 : acc0;
        acc = fmaf(rv.x, xv.x, acc);
        acc = fmaf(rv.y, xv.y, acc);
        acc = fmaf(rv.z, xv.z, acc);
        acc = fmaf(rv.w, xv.w, acc);
    }
    return acc0 + acc1;
}

// 1024 bf16 weights at w (smem) dotted with 1024 fp32 values at v (smem),
// summed over the warp.
__device__ __forceinline__ float bf16_dot1024(const __nv_bfloat16 *w, const float *v, int lane) {
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int c = 8 * (lane + 32 * i);
        const uint4 wv = *reinterpret_cast<const uint4 *>(w + c);
        float xv[8];
        *reinterpret_cast<float4 *>(xv) = *reinterpret_cast<const float4 *>(v + c);
        *reinterpret_cast<float4 *>(xv + 4) = *reinterpret_cast<const float4 *>(v + c + 4);
        if (i & 1) acc1 = dot8_bf16(wv, xv, acc1);
        else acc0 = dot8_bf16(wv, xv, acc0);
    }
    return warp_sum(acc0 + acc1);
}

__device__ __forceinline__ uint32_t bfe7(uint32_t v, uint32_t pos) {
    uint32_t r;
    asm("bfe.u32 %0, %1, %2, 7;" : "=r"(r) : "r"(v), "r"(pos));
    return r;
}

// One IQ2_XXS tile-block (16 rows x 256 cols) at tb, block column b, against
// the fp16 hi/lo activation: returns (in lanes t == 0) rows g and g+8.
// Lane (g, t) owns sub-blocks t and t+4 of rows g and g+8; the mma's B
// operand is block-diagonal (only lanes with g/2 == t feed x, the others read
// zeros), so each lane receives the sums of its own sub-blocks and applies
// its own scales.
__device__ __forceinline__ void iq2_tileblock(const D1Smem &sm, const uint8_t *tb, int b, int lane, float &r0,
                                              float &r1) {
    const int g = lane >> 2, t = lane & 3, p = lane & 15;
    const uint4 qa = *reinterpret_cast<const uint4 *>(tb + 16 * lane);
    const uint4 qb = *reinterpret_cast<const uint4 *>(tb + 512 + 16 * lane);
    const uint32_t dd = *reinterpret_cast<const uint32_t *>(tb + 1024 + 4 * g);
    const float d4g = __half2float(__ushort_as_half((unsigned short)(dd & 0xffffu))) * 4194304.0f;
    const float d4h = __half2float(__ushort_as_half((unsigned short)(dd >> 16))) * 4194304.0f;
    const __half *xb = ((g >> 1) == t) ? sm.xq + (g & 1) * kH + 256 * b + 32 * t : sm.zero;
    const uint2 *gt = sm.gtab + p, *st = sm.stab + (lane & 7);   // entry i at gt[16 i], st[8 i]
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
        uint32_t B[16];
        const uint4 *src = reinterpret_cast<const uint4 *>(xb + 128 * jj);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 v = src[q];
            B[4 * q + 0] = v.x;
            B[4 * q + 1] = v.y;
            B[4 * q + 2] = v.z;
            B[4 * q + 3] = v.w;
        }
        const uint32_t ia = jj ? qa.z : qa.x, va = jj ? qa.w : qa.y;
        const uint32_t ib = jj ? qb.z : qb.x, vb = jj ? qb.w : qb.y;
        // two independent accumulators so consecutive mma do not wait on each other
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int l = 0; l < 4; ++l) {
            const uint2 ga = gt[16 * __byte_perm(ia, 0, 0x4440 + l)];
            const uint2 gb = gt[16 * __byte_perm(ib, 0, 0x4440 + l)];
            const uint2 sa = st[8 * bfe7(va, 7 * l)];
            const uint2 sbv = st[8 * bfe7(vb, 7 * l)];
            mma_f16(c0, prmt(ga.x, sa.x, 0x5140), prmt(gb.x, sbv.x, 0x5140), prmt(ga.x, sa.x, 0x7362),
                    prmt(gb.x, sbv.x, 0x7362), B[4 * l], B[4 * l + 1]);
            mma_f16(c1, prmt(ga.y, sa.y, 0x5140), prmt(gb.y, sbv.y, 0x5140), prmt(ga.y, sa.y, 0x7362),
                    prmt(gb.y, sbv.y, 0x7362), B[4 * l + 2], B[4 * l + 3]);
        }
        acc0 = fmaf(d4g * half_plus(va >> 28), (c0[0] + c0[1]) + (c1[0] + c1[1]), acc0);
        acc1 = fmaf(d4h * half_plus(vb >> 28), (c0[2] + c0[3]) + (c1[2] + c1[3]), acc1);
    }
    acc0 += __shfl_xor_sync(0xffffffffu, acc0, 1);
    acc0 += __shfl_xor_sync(0xffffffffu, acc0, 2);
    acc1 += __shfl_xor_sync(0xffffffffu, acc1, 1);
    acc1 += __shfl_xor_sync(0xffffffffu, acc1, 2);
    r0 = acc0;
    r1 = acc1;
}

// Two adjacent IQ2_XXS tile-blocks (block columns b0, b0 + 1; 16 rows x 512
// cols) processed interleaved for instruction-level parallelism; returns the
// sum of both (in lanes t == 0) for rows g and g+8.  Same arithmetic as
// iq2_tileblock.
__device__ __forceinline__ void iq2_tileblock2(const D1Smem &sm, const uint8_t *tb, int b0, int lane, float &r0,
                                               float &r1) {
    const int g = lane >> 2, t = lane & 3, p = lane & 15;
    uint4 qa[2], qb[2];
    float d4g[2], d4h[2];
    const __half *xb[2];
    const bool act = (g >> 1) == t;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const uint8_t *tbu = tb + u * kTB_IQ2;
        qa[u] = *reinterpret_cast<const uint4 *>(tbu + 16 * lane);
        qb[u] = *reinterpret_cast<const uint4 *>(tbu + 512 + 16 * lane);
        const uint32_t dd = *reinterpret_cast<const uint32_t *>(tbu + 1024 + 4 * g);
        d4g[u] = __half2float(__ushort_as_half((unsigned short)(dd & 0xffffu))) * 4194304.0f;
        d4h[u] = __half2float(__ushort_as_half((unsigned short)(dd >> 16))) * 4194304.0f;
        xb[u] = act ? sm.xq + (g & 1) * kH + 256 * (b0 + u) + 32 * t : sm.zero;
    }
    const uint2 *gt = sm.gtab + p, *st = sm.stab + (lane & 7);   // entry i at gt[16 i], st[8 i]
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
        float c0[2][4], c1[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int i = 0; i < 4; ++i) c0[u][i] = c1[u][i] = 0.f;
#pragma unroll
        for (int l = 0; l < 4; ++l) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const uint4 B4 = *reinterpret_cast<const uint4 *>(xb[u] + 128 * jj + 8 * l);
                const uint32_t ia = jj ? qa[u].z : qa[u].x, va = jj ? qa[u].w : qa[u].y;
                const uint32_t ib = jj ? qb[u].z : qb[u].x, vb = jj ? qb[u].w : qb[u].y;
                const uint2 ga = gt[16 * __byte_perm(ia, 0, 0x4440 + l)];
                const uint2 gb = gt[16 * __byte_perm(ib, 0, 0x4440 + l)];
                const uint2 sa = st[8 * bfe7(va, 7 * l)];
                const uint2 sbv = st[8 * bfe7(vb, 7 * l)];
                mma_f16(c0[u], prmt(ga.x, sa.x, 0x5140), prmt(gb.x, sbv.x, 0x5140), prmt(ga.x, sa.x, 0x7362),
                        prmt(gb.x, sbv.x, 0x7362), B4.x, B4.y);
                mma_f16(c1[u], prmt(ga.y, sa.y, 0x5140), prmt(gb.y, sbv.y, 0x5140), prmt(ga.y, sa.y, 0x7362),
                        prmt(gb.y, sbv.y, 0x7362), B4.z, B4.w);
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const uint32_t va = jj ? qa[u].w : qa[u].y, vb = jj ? qb[u].w : qb[u].y;
            acc0 = fmaf(d4g[u] * half_plus(va >> 28), (c0[u][0] + c0[u][1]) + (c1[u][0] + c1[u][1]), acc0);
            acc1 = fmaf(d4h[u] * half_plus(vb >> 28), (c0[u][2] + c0[u][3]) + (c1[u][2] + c1[u][3]), acc1);
        }
    }
    acc0 += __shfl_xor_sync(0xffffffffu, acc0, 1);
    acc0 += __shfl_xor_sync(0xffffffffu, acc0, 2);
    acc1 += __shfl_xor_sync(0xffffffffu, acc1, 1);
    acc1 += __shfl_xor_sync(0xffffffffu, acc1, 2);
    r0 = acc0;
    r1 = acc1;
}

// One Q2_K tile-block (16 rows x 256 cols) of expert slot k, block column b,
// against h of slot k (fp16 hi/lo) and its 16-column sums.  Returns this
// lane's partial for rows g and g+8 (the quad's four lanes sum to the rows).
__device__ __forceinline__ void q2k_tileblock(const D1Smem &sm, const uint8_t *tb, int k, int b, int lane,
                                              float &s0, float &s1) {
    const int g = lane >> 2, t = lane & 3;
    const uint4 qa = *reinterpret_cast<const uint4 *>(tb + 16 * lane);
    const uint4 qb = *reinterpret_cast<const uint4 *>(tb + 512 + 16 * lane);
    const uint32_t sca = *reinterpret_cast<const uint32_t *>(tb + 1024 + 4 * lane);
    const uint32_t scb = *reinterpret_cast<const uint32_t *>(tb + 1152 + 4 * lane);
    const uint2 dd = *reinterpret_cast<const uint2 *>(tb + 1280 + 8 * g);
    const __half *hrow = ((g >> 1) == t) ? sm.hq + ((size_t)k * 2 + (g & 1)) * kF + 256 * b + 16 * t : sm.zero;
    const float4 X = *reinterpret_cast<const float4 *>(sm.xs16 + (size_t)k * 128 + (b * 4 + t) * 4);
    const float dg = __half2float(__ushort_as_half((unsigned short)(dd.x & 0xffff))) * 16777216.0f;
    const float mg = __half2float(__ushort_as_half((unsigned short)(dd.x >> 16)));
    const float dh = __half2float(__ushort_as_half((unsigned short)(dd.y & 0xffff))) * 16777216.0f;
    const float mh = __half2float(__ushort_as_half((unsigned short)(dd.y >> 16)));
    const uint32_t Wa[4] = {qa.x, qa.y, qa.z, qa.w};
    const uint32_t Wb[4] = {qb.x, qb.y, qb.z, qb.w};
    const float Xg[4] = {X.x, X.y, X.z, X.w};
    float sg = 0.f, sh = 0.f;
#pragma unroll
    for (int G = 0; G < 4; ++G) {
        float c[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
        uint4 hv[2];
        hv[0] = *reinterpret_cast<const uint4 *>(hrow + 64 * G);
        hv[1] = *reinterpret_cast<const uint4 *>(hrow + 64 * G + 8);
        const uint32_t hb[8] = {hv[0].x, hv[0].y, hv[0].z, hv[0].w, hv[1].x, hv[1].y, hv[1].z, hv[1].w};
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
            mma_f16((cc & 1) ? e : c, (Wa[G] >> (4 * cc)) & 0x00030003u, (Wb[G] >> (4 * cc)) & 0x00030003u,
                    (Wa[G] >> (4 * cc + 2)) & 0x00030003u, (Wb[G] >> (4 * cc + 2)) & 0x00030003u, hb[2 * cc],
                    hb[2 * cc + 1]);
        const uint32_t ba = (sca >> (8 * G)) & 0xffu, bb = (scb >> (8 * G)) & 0xffu;
        sg += dg * small_u2f(ba & 15u) * ((c[0] + c[1]) + (e[0] + e[1])) - mg * small_u2f(ba >> 4) * Xg[G];
        sh += dh * small_u2f(bb & 15u) * ((c[2] + c[3]) + (e[2] + e[3])) - mh * small_u2f(bb >> 4) * Xg[G];
    }
    s0 = sg;
    s1 = sh;
}

// Top-6 of the 256 router logits (sigmoid scores, bias for selection only,
// ties to the lower id, weights = selected scores renormalised), one warp.
// The result goes to this CTA's shared memory; CTA 0 also stores it for the
// caller.  bias_r: this lane's 8 bias values (experts lane + 32 i).
__device__ void d1_topk(const D1Args &a, const D1Smem &sm, const float (&bias_r)[8], int lane) {
    float key[8], s[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i] = __ldcg(a.logits + lane + 32 * i);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        s[i] = 1.0f / (1.0f + expf(-s[i]));
        key[i] = s[i] + bias_r[i];
    }
    int sel_e[kK];
    float sel_s[kK];
#pragma unroll
    for (int k = 0; k < kK; ++k) {
        float bk = -3.0e38f;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane + 32 * i;
            if (key[i] > bk || (key[i] == bk && e < be)) {
                bk = key[i];
                be = e;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ok = __shfl_xor_sync(0xffffffffu, bk, off);
            const int oe = __shfl_xor_sync(0xffffffffu, be, off);
            if (ok > bk || (ok == bk && oe < be)) {
                bk = ok;
                be = oe;
            }
        }
        const int owner = be & 31, slot = be >> 5;
        float sv = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i == slot) sv = s[i];
        sv = __shfl_sync(0xffffffffu, sv, owner);
        if (lane == owner) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i == slot) key[i] = -3.0e38f;
        }
        sel_e[k] = be;
        sel_s[k] = sv;
    }
    // the producer streams the selected experts' matrices: cache their
    // pointers here (one global load per pointer, once per CTA)
    if (lane < 3 * kK) {
        const int k = lane % kK, m = lane / kK;
        int e = 0;
#pragma unroll
        for (int kk = 0; kk < kK; ++kk)
            if (kk == k) e = sel_e[kk];
        const uint8_t *const *tab = m == 0 ? a.gate : m == 1 ? a.up : a.down;
        const uint8_t *ptr = tab[e];
        sm.eptr[lane] = (ptr && !((uintptr_t)ptr & 15)) ? ptr : nullptr;
    }
    __syncwarp();
    if (lane == 0) {
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < kK; ++k) sum += sel_s[k];
#pragma unroll
        for (int k = 0; k < kK; ++k) {
            const float wv = sel_s[k] / sum;
            sm.ids_s[k] = sel_e[k];
            sm.wk[k] = wv;
            if (blockIdx.x == 0) {
                a.ids[k] = sel_e[k];
                a.w[k] = wv;
            }
        }
        __threadfence_block();
        *reinterpret_cast<volatile int *>(&sm.flags[1]) = 1;
    }
}

// Jobs of phase p go to CTA (p even ? j : G-1-j) mod G.
__device__ __forceinline__ int phase_jobs(int p) {
    return p == 0 ? kJR : p == 1 ? kJSG : p == 2 ? kJSD : p == 3 ? kJRG : kJRD;
}
__device__ __forceinline__ int phase_off(int p, int c, int G) { return (p & 1) ? (G - 1 - c) : c; }
__device__ __forceinline__ int phase_pieces(int p) { return (p == 1 || p == 3) ? 2 : 1; }

// The CTA's i-th job -> (phase, job index); false past the end.
__device__ __forceinline__ bool cta_job(int i, int c, int G, const int (&cnt)[kNPhase], int &p, int &j) {
#pragma unroll
    for (int q = 0; q < kNPhase; ++q) {
        if (i < cnt[q]) {
            p = q;
            j = i * G + phase_off(q, c, G);
            return true;
        }
        i -= cnt[q];
    }
    return false;
}

// If this warp's counted job was the last of its 16-row output tile (the
// counter returned kTileParts - 1), sum the tile's partials in a fixed order:
// shared expert, then routed experts k = 0..5.
__device__ __forceinline__ void finish_tile(const D1Args &a, int tile, uint32_t old_lane0, int lane) {
    if (tile < 0) return;
    const uint32_t old = __shfl_sync(0xffffffffu, old_lane0, 0);
    if (old != kTileParts - 1) return;
    if (lane < 16) {
        const int row = 16 * tile + lane;
        float v = __ldcg(a.p_s + row);
#pragma unroll
        for (int k = 0; k < kK; ++k) v += __ldcg(a.p_r + (size_t)k * kH + row);
        a.out[row] = v;
    }
    if (lane == 0) a.sync->tile_cnt[tile] = 0u;
}

__global__ void __launch_bounds__(kD1Threads, 1) decode_t1_kernel(D1Args a) {
    const D1Smem sm = d1_smem();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, c = blockIdx.x;
    volatile int *abort_flag = sm.flags;
    if (tid == 0) {
        for (int i = 0; i < kD1Slots; ++i) {
            tc::mbar_init(&sm.full[i], 1);
            tc::mbar_init(&sm.empty[i], kGW);
        }
        sm.flags[0] = 0;
        sm.flags[1] = 0;
        sm.flags[2] = 0;
        tc::fence_mbar_init();
    }
    __syncthreads();
    int cnt[kNPhase];
#pragma unroll
    for (int p = 0; p < kNPhase; ++p) {
        const int off = phase_off(p, c, G), n = phase_jobs(p);
        cnt[p] = off < n ? (n - off + G - 1) / G : 0;
    }

    if (warp == 0) {
        // ================================================== producers
        // Lane q feeds group q's ring, so the four rings fill in parallel.
        if (lane < kNGrp) {
            const int q = lane;
            int gi = q, pcq = 0;
            uint32_t itq = 0;
            bool ids_known = false;
            long long t_idle = clock64();
            while (true) {
                if (*abort_flag) break;   // consumers leave on abort; nothing more to feed
                const int s = kSlotsPerGrp * q + (int)(itq % kSlotsPerGrp);
                if (!tc::mbar_test_wait(&sm.empty[s], ((itq / kSlotsPerGrp) & 1u) ^ 1u)) {
                    if (clock64() - t_idle > (2ll << 30)) {
                        // no slot freed for ~1 s: give up, let the groups finish
                        d1_abort(a, sm.flags, 0x11u);
                        break;
                    }
                    continue;
                }
                int p, j;
                if (!cta_job(gi, c, G, cnt, p, j)) {
                    sm.desc[s].kind = PK_END;
                    tc::mbar_arrive(&sm.full[s]);
                    break;
                }
                if ((p == 3 || p == 4) && !ids_known) {
                    if (*reinterpret_cast<volatile int *>(&sm.flags[1]) == 0) {   // later
                        if (clock64() - t_idle > (2ll << 30)) {
                            d1_abort(a, sm.flags, 0x12u);
                            break;
                        }
                        continue;
                    }
                    ids_known = true;
                }
                const int pc = pcq;
                uint8_t *dst = sm.ring + (size_t)s * kD1Slot;
                D1Desc d;
                d.job = j;
                d.piece = pc;
                d.e = 0;
                const void *src = nullptr;
                uint32_t bytes = 0;
                if (p == 0) {
                    d.kind = PK_ROUTER;
                    src = a.router + (size_t)j * kH;
                    bytes = kH * 4;
                } else if (p == 1) {
                    d.kind = PK_SGU;
                    src = (pc ? a.sh_up : a.sh_gate) + (size_t)(2 * j) * kH;
                    bytes = 2 * kH * 2;
                } else if (p == 2) {
                    d.kind = PK_SDN;
                    src = a.sh_down + (size_t)(4 * j) * kF;
                    bytes = 4 * kF * 2;
                } else if (p == 3) {
                    d.kind = PK_RGU;
                    const int k = j / (kF / 16), tile = j % (kF / 16);
                    const uint8_t *mat = sm.eptr[(pc ? kK : 0) + k];
                    d.e = k;
                    if (mat && sm.eptr[k] && sm.eptr[kK + k]) {
                        src = mat + (size_t)tile * 16 * kTB_IQ2;
                        bytes = 16 * kTB_IQ2;
                    } else {
                        d.e = -1;
                        flag_status(a.status, DS4G_EDEVICE, (uint32_t)sm.ids_s[k]);
                    }
                } else {
                    d.kind = PK_RDN;
                    const int k = j / (kH / 16), tile = j % (kH / 16);
                    const uint8_t *mat = sm.eptr[2 * kK + k];
                    d.e = k;
                    if (mat) {
                        src = mat + (size_t)tile * 8 * kTB_Q2K;
                        bytes = 8 * kTB_Q2K;
                    } else {
                        d.e = -1;
                        flag_status(a.status, DS4G_EDEVICE, (uint32_t)sm.ids_s[k]);
                    }
                }
                sm.desc[s] = d;
                if (bytes) {
                    tc::mbar_arrive_expect_tx(&sm.full[s], bytes);
                    bulk_load(dst, src, bytes, &sm.full[s]);
                } else {
                    tc::mbar_arrive(&sm.full[s]);
                }
                ++itq;
                if (++pcq == phase_pieces(p)) {
                    pcq = 0;
                    gi += kNGrp;
                }
                t_idle = clock64();
            }
        }
    } else if (warp == 1) {
        // ================================================== router warp
        float bias_r[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) bias_r[i] = __ldg(a.bias + lane + 32 * i);
        bool ok = true;
        if (lane == 0) ok = spin_geq(&a.sync->router_done, (uint32_t)kJR, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (ok) {
            d1_topk(a, sm, bias_r, lane);
        } else if (lane == 0) {
            d1_abort(a, sm.flags, 0x31u);
        }
    } else {
        // ================================================== consumers
        const int cw = warp - 2, ct = tid - 64;
        const int q = cw / kGW, wq = cw % kGW;
        // tables and the normalised activation (all 16 consumer warps); the
        // global loads are issued first, the tables built while they fly
        float xv[8], ss = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) xv[i] = __ldg(a.x + ct + 512 * i);
        const uint64_t grow = ct < 256 ? __ldg(reinterpret_cast<const unsigned long long *>(a.grid) + ct) : 0ull;
        for (int i = ct; i < 128 * 8; i += kD1Cons * 32) {
            const uint32_t s7 = (uint32_t)(i >> 3);
            const uint32_t sg = s7 | ((uint32_t)(__popc(s7) & 1) << 7);
            uint32_t lo = 0, hi = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                lo |= ((sg >> j) & 1u) << (8 * j + 7);
                hi |= ((sg >> (j + 4)) & 1u) << (8 * j + 7);
            }
            sm.stab[i] = make_uint2(lo, hi);
        }
        if (ct < 128) reinterpret_cast<uint32_t *>(sm.zero)[ct] = 0u;
        if (ct < 256) {
            const uint2 v = make_uint2((uint32_t)grow, (uint32_t)(grow >> 32));
#pragma unroll
            for (int rep = 0; rep < 16; ++rep) sm.gtab[ct * 16 + rep] = v;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(xv[i], xv[i], ss);
        ss = warp_sum(ss);
        if (lane == 0) sm.cta_red[cw] = ss;
        asm volatile("bar.sync 1, %0;" ::"n"(kD1Cons * 32));
        float tot = 0.f;
#pragma unroll
        for (int i = 0; i < kD1Cons; ++i) tot += sm.cta_red[i];
        const float r = a.normalize ? 1.0f / sqrtf(tot * (1.0f / kH) + 1e-6f) : 1.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float v = xv[i] * r;
            if (!(fabsf(v) < 65504.f)) flag_status(a.status, DS4G_EDEVICE, 0xF16u);
            sm.xn[ct + 512 * i] = v;
            __half hi, lo;
            split_f16(v, hi, lo);
            sm.xq[ct + 512 * i] = hi;
            sm.xq[kH + ct + 512 * i] = lo;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kD1Cons * 32));

        float rg0 = 0.f, rg1 = 0.f, ru0 = 0.f, ru1 = 0.f; // routed gate/up partials, rows g, g+8
        int pend_tile = -1;                               // tile counted by this warp, not yet examined
        uint32_t pend_old = 0u;
        bool in_down = false;
        int gpar = 0;
        for (uint32_t it = 0;; ++it) {
            const int s = kSlotsPerGrp * q + (int)(it % kSlotsPerGrp);
            if (!d1_wait(&sm.full[s], (it / kSlotsPerGrp) & 1u, abort_flag)) {
                d1_abort(a, sm.flags, 0x21u);
                // still take part in the CTA transition below so no barrier is left waiting
                if (!in_down) {
                    asm volatile("bar.sync 1, %0;" ::"n"(kD1Cons * 32));
                    asm volatile("bar.sync 1, %0;" ::"n"(kD1Cons * 32));
                    asm volatile("bar.sync 1, %0;" ::"n"(kD1Cons * 32));
                }
                break;
            }
            const D1Desc d = sm.desc[s];
            if (!in_down && (d.kind == PK_END || d.kind == PK_RDN)) {
                // This group has no routed gate/up work left.  Once all four groups
                // are here, publish this CTA's routed h, wait for every CTA's, then
                // load it (over the gate/up tables, which are no longer needed).
                asm volatile("bar.sync 1, %0;" ::"n"(kD1Cons * 32));
                if (ct == 0) {
                    red_add_release(&a.sync->gu_cta, 1u);
                    if (!spin_geq(&a.sync->gu_cta, (uint32_t)G, abort_flag)) d1_abort(a, sm.flags, 0x22u);
                }
                asm volatile("bar.sync 1, %0;" ::"n"(kD1Cons * 32));
                {
                    // h of the six slots: 768 groups of 16 columns; thread ct takes
                    // groups ct and ct + 512 (all loads issued first)
                    float4 hv[2][4];
                    const float4 *h4 = reinterpret_cast<const float4 *>(a.h_r);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int grp = ct + 512 * u;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            hv[u][j] = grp < kK * 128 ? __ldcg(h4 + 4 * grp + j) : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int grp = ct + 512 * u;
                        if (grp >= kK * 128) continue;
                        const int k = grp >> 7, gl = grp & 127;
                        const float hf[16] = {hv[u][0].x, hv[u][0].y, hv[u][0].z, hv[u][0].w,
                                              hv[u][1].x, hv[u][1].y, hv[u][1].z, hv[u][1].w,
                                              hv[u][2].x, hv[u][2].y, hv[u][2].z, hv[u][2].w,
                                              hv[u][3].x, hv[u][3].y, hv[u][3].z, hv[u][3].w};
                        float sum = 0.f;
                        uint32_t hi2[8], lo2[8];
#pragma unroll
                        for (int j = 0; j < 16; j += 2) {
                            sum += hf[j] + hf[j + 1];
                            __half h0, l0, h1, l1;
                            split_f16(hf[j], h0, l0);
                            split_f16(hf[j + 1], h1, l1);
                            hi2[j / 2] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
                            lo2[j / 2] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
                        }
                        uint4 *dh = reinterpret_cast<uint4 *>(sm.hq + ((size_t)k * 2) * kF + 16 * gl);
                        uint4 *dl = reinterpret_cast<uint4 *>(sm.hq + ((size_t)k * 2 + 1) * kF + 16 * gl);
                        dh[0] = make_uint4(hi2[0], hi2[1], hi2[2], hi2[3]);
                        dh[1] = make_uint4(hi2[4], hi2[5], hi2[6], hi2[7]);
                        dl[0] = make_uint4(lo2[0], lo2[1], lo2[2], lo2[3]);
                        dl[1] = make_uint4(lo2[4], lo2[5], lo2[6], lo2[7]);
                        const int b = gl >> 4, j16 = gl & 15;
                        sm.xs16[k * 128 + (b * 4 + (j16 & 3)) * 4 + (j16 >> 2)] = sum;
                    }
                }
                asm volatile("bar.sync 1, %0;" ::"n"(kD1Cons * 32));
                in_down = true;
            }
            if (d.kind == PK_END) break;
            if (d.kind == PK_SDN && *reinterpret_cast<volatile int *>(&sm.flags[2]) != 2) {
                // first shared-down piece of this CTA: one group waits until every
                // shared gate/up row is stored and loads shared h; others wait for it
                int role = 0;
                if (lane == 0 && wq == 0) role = atomicCAS(&sm.flags[2], 0, 1) == 0 ? 1 : 0;
                role = __shfl_sync(0xffffffffu, role, 0);
                role = __shfl_sync(0xffffffffu, role, 0);
                asm volatile("bar.sync %0, %1;" ::"r"(2 + q), "n"(kGW * 32));
                // broadcast the group's decision through shared memory
                if (wq == 0 && lane == 0) sm.cta_red[q] = role ? 1.f : 0.f;
                asm volatile("bar.sync %0, %1;" ::"r"(2 + q), "n"(kGW * 32));
                const bool loader = sm.cta_red[q] != 0.f;
                if (loader) {
                    if (wq == 0 && lane == 0 && !spin_geq(&a.sync->sgu_done, (uint32_t)kJSG, abort_flag))
                        d1_abort(a, sm.flags, 0x23u);
                    asm volatile("bar.sync %0, %1;" ::"r"(2 + q), "n"(kGW * 32));
                    const int gt = wq * 32 + lane;   // 128 threads x 4 float4
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        reinterpret_cast<float4 *>(sm.hs)[gt + 128 * u] =
                            __ldcg(reinterpret_cast<const float4 *>(a.h_s) + gt + 128 * u);
                    __threadfence_block();
                    asm volatile("bar.sync %0, %1;" ::"r"(2 + q), "n"(kGW * 32));
                    if (wq == 0 && lane == 0) *reinterpret_cast<volatile int *>(&sm.flags[2]) = 2;
                } else {
                    const long long t0 = clock64();
                    while (*reinterpret_cast<volatile int *>(&sm.flags[2]) != 2 && !*abort_flag) {
                        if (clock64() - t0 > (2ll << 30)) {
                            d1_abort(a, sm.flags, 0x24u);
                            break;
                        }
                        __nanosleep(64);
                    }
                    __threadfence_block();
                }
            }
            const uint8_t *slot = sm.ring + (size_t)s * kD1Slot;
            float *red = sm.red + (q * 2 + gpar) * 128;
            bool last = false;
            if (d.kind == PK_ROUTER) {
                // router row: warp wq takes columns [1024 wq, +1024)
                const float v = warp_sum(router_row(sm, slot, wq, lane));
                if (lane == 0) red[wq] = v;
                last = true;
            } else if (d.kind == PK_SGU) {
                // piece 0: gate rows 2j, 2j+1; piece 1: up rows; warp wq: row wq>>1, half wq&1
                const __nv_bfloat16 *w = reinterpret_cast<const __nv_bfloat16 *>(slot) + (wq >> 1) * kH + 2048 * (wq & 1);
                const float *xv = sm.xn + 2048 * (wq & 1);
                const float v = bf16_dot1024(w, xv, lane) + bf16_dot1024(w + 1024, xv + 1024, lane);
                if (lane == 0) red[4 * d.piece + wq] = v;
                last = d.piece == 1;
            } else if (d.kind == PK_RGU) {
                if (d.piece == 0) rg0 = rg1 = ru0 = ru1 = 0.f;
                if (d.e >= 0) {
                    float t0, t1, t2, t3;
                    iq2_tileblock2(sm, slot + (size_t)(4 * wq) * kTB_IQ2, 4 * wq, lane, t0, t1);
                    iq2_tileblock2(sm, slot + (size_t)(4 * wq + 2) * kTB_IQ2, 4 * wq + 2, lane, t2, t3);
                    if (d.piece) {
                        ru0 += t0 + t2;
                        ru1 += t1 + t3;
                    } else {
                        rg0 += t0 + t2;
                        rg1 += t1 + t3;
                    }
                }
                if (d.piece == 1) {
                    if ((lane & 3) == 0) {
                        red[wq * 16 + (lane >> 2)] = rg0;
                        red[wq * 16 + (lane >> 2) + 8] = rg1;
                        red[64 + wq * 16 + (lane >> 2)] = ru0;
                        red[64 + wq * 16 + (lane >> 2) + 8] = ru1;
                    }
                    last = true;
                }
            } else if (d.kind == PK_SDN) {
                // shared down rows 4j .. 4j+3; warp wq: row wq, all 2048 columns
                const __nv_bfloat16 *w = reinterpret_cast<const __nv_bfloat16 *>(slot) + (size_t)wq * kF;
                const float v = bf16_dot1024(w, sm.hs, lane) + bf16_dot1024(w + 1024, sm.hs + 1024, lane);
                if (lane == 0) red[wq] = v;
                last = true;
            } else {  // PK_RDN: eight Q2_K tile-blocks of one expert; warp wq: tile-blocks 2wq, 2wq+1
                float s0 = 0.f, s1 = 0.f;
                if (d.e >= 0) {
                    float a0, a1, b0, b1;
                    q2k_tileblock(sm, slot + (size_t)(2 * wq) * kTB_Q2K, d.e, 2 * wq, lane, a0, a1);
                    q2k_tileblock(sm, slot + (size_t)(2 * wq + 1) * kTB_Q2K, d.e, 2 * wq + 1, lane, b0, b1);
                    s0 = a0 + b0;
                    s1 = a1 + b1;
                }
                s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
                s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
                s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
                s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
                if ((lane & 3) == 0) {
                    red[wq * 16 + (lane >> 2)] = s0;
                    red[wq * 16 + (lane >> 2) + 8] = s1;
                }
                last = true;
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&sm.empty[s]);
            if (!last) continue;
            // ---- job end: the group's four warps reduce in a fixed order
            asm volatile("bar.sync %0, %1;" ::"r"(2 + q), "n"(kGW * 32));
            if (wq == 0) {
                int tile = -1;
                if (d.kind == PK_ROUTER) {
                    if (lane == 0) {
                        a.logits[d.job] = (red[0] + red[1]) + (red[2] + red[3]);
                        red_add_release(&a.sync->router_done, 1u);
                    }
                } else if (d.kind == PK_SGU) {
                    if (lane < 2) {
                        a.h_s[2 * d.job + lane] = silu_f(red[2 * lane] + red[2 * lane + 1]) *
                                                  (red[4 + 2 * lane] + red[4 + 2 * lane + 1]);
                    }
                    __syncwarp();
                    if (lane == 0) red_add_release(&a.sync->sgu_done, 1u);
                } else if (d.kind == PK_RGU) {
                    if (lane < 16) {
                        const float gs = (red[lane] + red[16 + lane]) + (red[32 + lane] + red[48 + lane]);
                        const float us = (red[64 + lane] + red[80 + lane]) + (red[96 + lane] + red[112 + lane]);
                        const int k = d.job / (kF / 16), tl = d.job % (kF / 16);
                        a.h_r[(size_t)k * kF + 16 * tl + lane] = silu_f(gs) * us;
                    }
                } else if (d.kind == PK_SDN) {
                    if (lane < 4) a.p_s[4 * d.job + lane] = red[lane];
                    tile = (4 * d.job) / 16;
                } else {  // routed down partial of one expert, weighted
                    const int k = d.job / (kH / 16), tl = d.job % (kH / 16);
                    if (lane < 16) {
                        const float v = (red[lane] + red[16 + lane]) + (red[32 + lane] + red[48 + lane]);
                        a.p_r[(size_t)k * kH + 16 * tl + lane] = d.e >= 0 ? sm.wk[k] * v : 0.f;
                    }
                    tile = tl;
                }
                if (tile >= 0) {
                    // Count this job into its output tile; the last of the tile's 14
                    // jobs sums the partials.  The counter's old value is examined
                    // only at this warp's next job end, so its latency is hidden.
                    finish_tile(a, pend_tile, pend_old, lane);
                    __syncwarp();
                    pend_old = 0u;
                    if (lane == 0) pend_old = atom_add_acq_rel(&a.sync->tile_cnt[tile], 1u);
                    pend_tile = tile;
                }
            }
            gpar ^= 1;
        }
        if (wq == 0) finish_tile(a, pend_tile, pend_old, lane);
    }

    // ================================================== exit protocol
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const uint32_t done = atomicAdd(&a.sync->exit_count, 1u);
        if (done == gridDim.x - 1) {
            // every CTA has finished: reset the coordination block for the next launch
            a.sync->router_done = 0;
            a.sync->sgu_done = 0;
            a.sync->gu_cta = 0;
            for (int t = 0; t < kH / 16; ++t) a.sync->tile_cnt[t] = 0;   // already zero unless a launch gave up
            __threadfence();
            a.sync->exit_count = 0;
        }
    }
}

// ------------------------------------------------------------------ host
struct D1Layout {
    size_t sync, logits, h_r, h_s, p_s, p_r, total;
};
static D1Layout d1_layout() {
    D1Layout L;
    size_t off = kWsHeader;
    L.sync = off;
    off += align_up(sizeof(D1Sync), 256);
    L.logits = off;
    off += align_up(kE * 4, 256);
    L.h_r = off;
    off += align_up((size_t)kK * kF * 4, 256);
    L.h_s = off;
    off += align_up((size_t)kF * 4, 256);
    L.p_s = off;
    off += align_up((size_t)kH * 4, 256);
    L.p_r = off;
    off += align_up((size_t)kK * kH * 4, 256);
    L.total = off;
    return L;
}

static int g_d1_sms = 0;
static bool g_d1_attr = false;

}  // namespace ds4g

using namespace ds4g;

extern "C" size_t ds4g_layer_decode_workspace(void) { return d1_layout().total; }

extern "C" ds4g_status ds4g_moe_layer_decode(const float *hidden, int normalize, const float *router,
                                             const float *bias, const ds4g_layer *L, int32_t *ids, float *w,
                                             float *out, void *workspace, size_t ws_bytes, ds4g_stream_t s) {
    if (!hidden || !router || !bias || !L || !ids || !w || !out || !workspace) return DS4G_EINVAL;
    if (!L->gate || !L->up || !L->down || !L->sh_gate || !L->sh_up || !L->sh_down) return DS4G_EINVAL;
    if (L->gate_up_type != DS4G_IQ2_XXS || L->down_type != DS4G_Q2_K) return DS4G_EUNSUPPORTED;
    if (!L->iq2_grid) return DS4G_EINVAL;
    const uintptr_t al = (uintptr_t)hidden | (uintptr_t)router | (uintptr_t)bias | (uintptr_t)ids |
                         (uintptr_t)w | (uintptr_t)out | (uintptr_t)workspace | (uintptr_t)L->gate |
                         (uintptr_t)L->up | (uintptr_t)L->down | (uintptr_t)L->sh_gate | (uintptr_t)L->sh_up |
                         (uintptr_t)L->sh_down | (uintptr_t)L->iq2_grid;
    if (al & 15) return DS4G_EALIGN;
    const D1Layout lay = d1_layout();
    if (ws_bytes < lay.total) return DS4G_ENOSPACE;
    if (!g_d1_sms) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return DS4G_ECUDA;
        if (cudaDeviceGetAttribute(&g_d1_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DS4G_ECUDA;
    }
    if (!g_d1_attr) {
        if (cudaFuncSetAttribute(decode_t1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kD1SmemBytes) !=
            cudaSuccess)
            return DS4G_ECUDA;
        g_d1_attr = true;
    }
    uint8_t *ws = (uint8_t *)workspace;
    D1Args a;
    a.x = hidden;
    a.normalize = normalize ? 1 : 0;
    a.router = router;
    a.bias = bias;
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
    a.status = (uint32_t *)ws;
    a.sync = (D1Sync *)(ws + lay.sync);
    a.logits = (float *)(ws + lay.logits);
    a.h_r = (float *)(ws + lay.h_r);
    a.h_s = (float *)(ws + lay.h_s);
    a.p_s = (float *)(ws + lay.p_s);
    a.p_r = (float *)(ws + lay.p_r);
    decode_t1_kernel<<<g_d1_sms, kD1Threads, kD1SmemBytes, (cudaStream_t)s>>>(a);
    return cudaGetLastError() == cudaSuccess ? DS4G_OK : DS4G_ECUDA;
}
