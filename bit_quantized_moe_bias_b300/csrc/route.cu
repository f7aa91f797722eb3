// route.cu — router scores and top-6 selection (chenxutan ds4 article §3.2
// "Router 计算专家选择"; juejin ds4 article §2.1: 256 routed experts, 6 used).
// Readings where the pages are silent: sigmoid score, bias only for
// selection, ties to the lower expert id, weights = selected unbiased scores
// renormalised to sum 1.
//
// One launch for any T:
//   small T (<= 8): CTA (expert group of 8, k-quarter); each warp streams one
//     router row quarter once and dots it with all T tokens (4 at a time);
//   mid T (9..64): CTA (expert group of 16, 512-column k-slice) with the
//     slice of x and of R staged in shared memory, one lane per token; a
//     second launch runs the top-6, one warp per token;
//   large T: 32-token x 64-expert fp32 SIMT tiles over a quarter of K each
//     (the whole K above 16384 tokens).
// Partial logits go to the workspace; the last CTA to finish a token range
// (atomic ticket, no waiting) sums them in a fixed order and runs the top-k,
// one warp per token.
#include <float.h>

#include "ds4g_internal.cuh"

namespace ds4g {

constexpr int kRouteSmallT = 64;
constexpr int kRouteKS = 4;   // k-splits on the small-T path
constexpr int kRouteFusedTopK = 8;   // up to here: the small-T path, whose last CTA runs the top-6
constexpr int kMidKS = 8;            // k-splits on the mid-T path
constexpr int kMidKC = kH / kMidKS;  // 512 columns per split
constexpr int kMidE = 16;            // experts per CTA (4 warps x 4)
constexpr int kMidXLd = kMidKC + 4;  // x row in shared memory (+16 B: rows start on distinct banks)
constexpr int kTileT = 32, kTileE = 64, kTileK = 32;

struct RouteArgs {
    const float *x;
    int T;
    const float *R;
    const float *bias;
    int32_t *ids;
    float *w;
    float *part;      // small / mid: [KS][T][256]; large: [T][256]
    int nks;          // k-splits summed by route_topk_kernel
    uint32_t *cnt;    // small: [1]; large: [ceil(T/32)]
    uint32_t *status;
};

// Warp: top-6 for one token given its 256 logits (in shared memory).
__device__ void topk_warp(const RouteArgs &a, int t, const float *logit) {
    const int lane = threadIdx.x & 31;
    float key[8], s[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i;
        s[i] = 1.0f / (1.0f + expf(-logit[e]));
        key[i] = s[i] + a.bias[e];
    }
    int sel_e[kK];
    float sel_s[kK];
#pragma unroll
    for (int k = 0; k < kK; ++k) {
        float bk = -FLT_MAX;
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
                if (i == slot) key[i] = -FLT_MAX;
        }
        sel_e[k] = be;
        sel_s[k] = sv;
    }
    if (lane == 0) {
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < kK; ++k) sum += sel_s[k];
#pragma unroll
        for (int k = 0; k < kK; ++k) {
            a.ids[t * kK + k] = sel_e[k];
            a.w[t * kK + k] = sel_s[k] / sum;
        }
    }
}

// grid (32, KS), block 256.
__global__ void __launch_bounds__(256) route_small_kernel(RouteArgs a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * 8 + warp, ks = blockIdx.y;
    const int k0 = ks * (kH / kRouteKS);
    float4 r[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        r[i] = __ldcs(reinterpret_cast<const float4 *>(a.R + (size_t)e * kH + k0 + 4 * lane + 128 * i));
    for (int t0 = 0; t0 < a.T; t0 += 4) {
        // four tokens at a time: their activation loads are in flight together
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (t0 + u >= a.T) break;
            const float *xr = a.x + (size_t)(t0 + u) * kH + k0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 xv = __ldg(reinterpret_cast<const float4 *>(xr + 4 * lane + 128 * i));
                acc[u] = fmaf(r[i].x, xv.x, acc[u]);
                acc[u] = fmaf(r[i].y, xv.y, acc[u]);
                acc[u] = fmaf(r[i].z, xv.z, acc[u]);
                acc[u] = fmaf(r[i].w, xv.w, acc[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float v = acc[u];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == 0 && t0 + u < a.T) a.part[((size_t)ks * a.T + t0 + u) * kE + e] = v;
        }
    }
    __threadfence();  // every writer publishes its partials before the ticket
    __shared__ uint32_t last;
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t ticket = atomicAdd(a.cnt, 1u);
        last = (ticket == gridDim.x * gridDim.y - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    // one warp per token: its logits (sum of the k-quarters in order), top-6
    __shared__ float lg[8][kE];
    for (int t = warp; t < a.T; t += 8) {
        for (int ee = lane; ee < kE; ee += 32) {
            float v = 0.f;
            for (int s = 0; s < kRouteKS; ++s) v += __ldcg(a.part + ((size_t)s * a.T + t) * kE + ee);
            lg[warp][ee] = v;
        }
        __syncwarp();
        topk_warp(a, t, lg[warp]);
        __syncwarp();
    }
    if (threadIdx.x == 0) *a.cnt = 0u;
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
                 "l"(gmem)
                 : "memory");
}

// Mid-T path: grid (256 / 16, 8), block 128, dynamic shared memory
// route_mid_smem(T).  CTA (g, ks) stages x[:, 512 ks .. +512] and the 16
// router rows 16 g .. +16 over the same columns, then lane l of warp w dots
// token l (and l + 32) with rows 16 g + 4 w .. +3: per row two interleaved
// accumulators over alternate 4-column steps, added at the end.  Partials
// part[ks][t][e].
__global__ void __launch_bounds__(128) route_mid_kernel(RouteArgs a) {
    extern __shared__ __align__(16) float msm[];
    float *xs = msm;                                // [T][kMidXLd]
    float *rs = msm + (size_t)a.T * kMidXLd;        // [16][kMidKC]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int e0 = blockIdx.x * kMidE, ks = blockIdx.y, k0 = ks * kMidKC;
    constexpr int kC4 = kMidKC / 4;                 // 16-byte chunks per row slice
    for (int i = tid; i < a.T * kC4; i += 128) {
        const int t = i / kC4, c4 = i % kC4;
        cp_async16(xs + (size_t)t * kMidXLd + 4 * c4, a.x + (size_t)t * kH + k0 + 4 * c4);
    }
    for (int i = tid; i < kMidE * kC4; i += 128) {
        const int e = i / kC4, c4 = i % kC4;
        cp_async16(rs + (size_t)e * kMidKC + 4 * c4, a.R + (size_t)(e0 + e) * kH + k0 + 4 * c4);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    const float *rr = rs + (size_t)(4 * warp) * kMidKC;
    for (int tb = 0; tb < a.T; tb += 32) {
        const int t = tb + lane;
        const bool has = t < a.T;
        const float *xr = xs + (size_t)(has ? t : 0) * kMidXLd;
        float acc[4][2];
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = 0.f;
#pragma unroll 2
        for (int k = 0; k < kMidKC; k += 8) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float4 xv = *reinterpret_cast<const float4 *>(xr + k + 4 * h);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 rv = *reinterpret_cast<const float4 *>(rr + (size_t)j * kMidKC + k + 4 * h);
                    float v = acc[j][h];
                    v = fmaf(rv.x, xv.x, v);
                    v = fmaf(rv.y, xv.y, v);
                    v = fmaf(rv.z, xv.z, v);
                    v = fmaf(rv.w, xv.w, v);
                    acc[j][h] = v;
                }
            }
        }
        if (has)
            *reinterpret_cast<float4 *>(a.part + ((size_t)ks * a.T + t) * kE + e0 + 4 * warp) =
                make_float4(acc[0][0] + acc[0][1], acc[1][0] + acc[1][1], acc[2][0] + acc[2][1],
                            acc[3][0] + acc[3][1]);
    }
}

// Mid-T path: the top-6 of each token from the k-split partials (summed in
// order), one warp per token, ceil(T/8) CTAs.
__global__ void __launch_bounds__(256) route_topk_kernel(RouteArgs a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    __shared__ float lg[8][kE];
    if (t >= a.T) return;
    // logit ee = lane + 32 i: the splits added in order; the loads of a
    // split are independent of each other and of the previous split's adds
    float v[kE / 32];
#pragma unroll
    for (int i = 0; i < kE / 32; ++i) v[i] = 0.f;
#pragma unroll 4
    for (int s = 0; s < a.nks; ++s) {
        float p[kE / 32];
#pragma unroll
        for (int i = 0; i < kE / 32; ++i) p[i] = __ldcg(a.part + ((size_t)s * a.T + t) * kE + lane + 32 * i);
#pragma unroll
        for (int i = 0; i < kE / 32; ++i) v[i] += p[i];
    }
#pragma unroll
    for (int i = 0; i < kE / 32; ++i) lg[warp][lane + 32 * i] = v[i];
    __syncwarp();
    topk_warp(a, t, lg[warp]);
}

// grid (ceil(T/32), 4, nks), block 128: fp32 tile 32 tokens x 64 experts over
// k-slice blockIdx.z of nks; thread (ty, tx) accumulates tokens 4ty..4ty+3 x
// experts 4tx..4tx+3 (16 FMA per two 16-byte shared loads).  Tiles are stored
// k-major; the next K chunk is loaded into registers while the current one is
// multiplied.  Partials part[z][t][e]; the last of the token tile's 4 x nks
// CTAs adds the slices in order and runs the top-6 of its 32 tokens.
constexpr int kRouteTiledThreads = 128;
__global__ void __launch_bounds__(kRouteTiledThreads) route_tiled_kernel(RouteArgs a) {
    __shared__ __align__(16) float xs[2][kTileK][kTileT];
    __shared__ __align__(16) float rs[2][kTileK][kTileE];
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const int t0 = blockIdx.x * kTileT, e0 = blockIdx.y * kTileE;
    const int kn = kH / a.nks, kb0 = blockIdx.z * kn;   // this CTA's k-slice
    // global -> register staging: x tile 32 x 32 (2 float4 per thread), R tile 64 x 32 (4)
    float4 xr[2], rr[4];
    auto load = [&](int k0) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = tid + kRouteTiledThreads * u, tt = i >> 3, kq = i & 7;
            xr[u] = (t0 + tt < a.T) ? __ldg(reinterpret_cast<const float4 *>(a.x + (size_t)(t0 + tt) * kH + k0) + kq)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = tid + kRouteTiledThreads * u, ee = i >> 3, kq = i & 7;
            rr[u] = __ldg(reinterpret_cast<const float4 *>(a.R + (size_t)(e0 + ee) * kH + k0) + kq);
        }
    };
    auto store = [&](int buf) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = tid + kRouteTiledThreads * u, tt = i >> 3, k = 4 * (i & 7);
            xs[buf][k][tt] = xr[u].x;
            xs[buf][k + 1][tt] = xr[u].y;
            xs[buf][k + 2][tt] = xr[u].z;
            xs[buf][k + 3][tt] = xr[u].w;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = tid + kRouteTiledThreads * u, ee = i >> 3, k = 4 * (i & 7);
            rs[buf][k][ee] = rr[u].x;
            rs[buf][k + 1][ee] = rr[u].y;
            rs[buf][k + 2][ee] = rr[u].z;
            rs[buf][k + 3][ee] = rr[u].w;
        }
    };
    float acc[4][4] = {};
    load(kb0);
    store(0);
    __syncthreads();
    int buf = 0;
    for (int k0 = kb0; k0 < kb0 + kn; k0 += kTileK) {
        const bool more = k0 + kTileK < kb0 + kn;
        if (more) load(k0 + kTileK);
#pragma unroll 8
        for (int kk = 0; kk < kTileK; ++kk) {
            const float4 xv = *reinterpret_cast<const float4 *>(&xs[buf][kk][4 * ty]);
            const float4 rv = *reinterpret_cast<const float4 *>(&rs[buf][kk][4 * tx]);
            const float xa[4] = {xv.x, xv.y, xv.z, xv.w}, ra[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xa[i], ra[j], acc[i][j]);
        }
        if (more) store(buf ^ 1);
        __syncthreads();
        buf ^= 1;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = t0 + 4 * ty + i;
        if (t < a.T)
            *reinterpret_cast<float4 *>(a.part + ((size_t)blockIdx.z * a.T + t) * kE + e0 + 4 * tx) =
                make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    }
    __threadfence();
    __shared__ uint32_t last;
    __syncthreads();
    if (tid == 0) {
        const uint32_t ticket = atomicAdd(a.cnt + blockIdx.x, 1u);
        last = (ticket == gridDim.y * gridDim.z - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    constexpr int kW = kRouteTiledThreads / 32;
    __shared__ float lg[kW][kE];
    const int warp = tid >> 5, lane = tid & 31;
    for (int tt = warp; tt < kTileT; tt += kW) {
        const int t = t0 + tt;
        if (t >= a.T) break;
        for (int i = lane; i < kE; i += 32) {
            float v = 0.f;
            for (int z = 0; z < a.nks; ++z) v += __ldcg(a.part + ((size_t)z * a.T + t) * kE + i);
            lg[warp][i] = v;
        }
        __syncwarp();
        topk_warp(a, t, lg[warp]);
        __syncwarp();
    }
    if (tid == 0) a.cnt[blockIdx.x] = 0u;
}

}  // namespace ds4g

using namespace ds4g;

// k-slices of the tiled path: 4 up to kTiledSplitMaxT tokens (more CTAs for
// the SMs), 1 beyond (the partials would grow to 4 KB per token)
constexpr int kTiledSplitMaxT = 16384;
static int tiled_nks(int T) { return T <= kTiledSplitMaxT ? 4 : 1; }

static size_t route_part_bytes(int T) {
    if (T <= kRouteFusedTopK) return (size_t)kRouteKS * T * kE * 4;
    if (T <= kRouteSmallT) return (size_t)kMidKS * T * kE * 4;
    return (size_t)tiled_nks(T) * T * kE * 4;
}

static size_t route_mid_smem(int T) { return ((size_t)T * kMidXLd + (size_t)kMidE * kMidKC) * 4; }

// Ticket counters at a fixed offset, sized for DS4G_ROUTE_MAX_T tokens, so
// that a workspace reused with another T never finds old partials where its
// (zero) counters should be; partials after them.
constexpr size_t kRouteCntBytes = ((size_t)(DS4G_ROUTE_MAX_T / kTileT + 1) * 4 + 255) / 256 * 256;

static size_t route_ws_need(int T) { return kWsHeader + kRouteCntBytes + align_up(route_part_bytes(T), 256); }

// The most any call with 1..T tokens needs: the partials of each path grow
// with T, so the maximum is over T and the largest T of every path below it.
extern "C" size_t ds4g_route_workspace(int T) {
    if (T < 1 || T > DS4G_ROUTE_MAX_T) return 0;
    size_t n = route_ws_need(T);
    const int tops[3] = {kRouteFusedTopK, kRouteSmallT, kTiledSplitMaxT};
    for (int i = 0; i < 3; ++i)
        if (tops[i] < T && route_ws_need(tops[i]) > n) n = route_ws_need(tops[i]);
    return n;
}

extern "C" ds4g_status ds4g_moe_route(const float *hidden, int T, const float *router,
                                      const float *bias, int32_t *ids, float *w, void *workspace,
                                      size_t ws_bytes, ds4g_stream_t s) {
    DS4G_TRACE();
    if (!hidden || !router || !bias || !ids || !w || !workspace || T < 1) return DS4G_EINVAL;
    if (T > DS4G_ROUTE_MAX_T) return DS4G_EUNSUPPORTED;
    if (((uintptr_t)hidden | (uintptr_t)router | (uintptr_t)bias | (uintptr_t)ids | (uintptr_t)w |
         (uintptr_t)workspace) & 15)
        return DS4G_EALIGN;
    if (ws_bytes < route_ws_need(T)) return DS4G_ENOSPACE;
    RouteArgs a;
    a.x = hidden;
    a.T = T;
    a.R = router;
    a.bias = bias;
    a.ids = ids;
    a.w = w;
    uint8_t *ws = (uint8_t *)workspace;
    a.status = (uint32_t *)ws;
    const size_t ntile = (size_t)(T + kTileT - 1) / kTileT;
    a.cnt = (uint32_t *)(ws + kWsHeader);
    a.part = (float *)(ws + kWsHeader + kRouteCntBytes);
    cudaStream_t st = (cudaStream_t)s;
    if (T <= kRouteFusedTopK) {
        a.nks = kRouteKS;
        route_small_kernel<<<dim3(kE / 8, kRouteKS), 256, 0, st>>>(a);
    } else if (T <= kRouteSmallT) {
        static bool attr = false;   // the largest mid-T staging (T = 64) once per process
        if (!attr) {
            if (cudaFuncSetAttribute(route_mid_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)route_mid_smem(kRouteSmallT)) != cudaSuccess)
                return DS4G_ECUDA;
            attr = true;
        }
        a.nks = kMidKS;
        route_mid_kernel<<<dim3(kE / kMidE, kMidKS), 128, route_mid_smem(T), st>>>(a);
        route_topk_kernel<<<(T + 7) / 8, 256, 0, st>>>(a);
    } else {
        a.nks = tiled_nks(T);
        route_tiled_kernel<<<dim3((unsigned)ntile, kE / kTileE, (unsigned)a.nks), kRouteTiledThreads, 0, st>>>(a);
    }
    return cudaGetLastError() == cudaSuccess ? DS4G_OK : DS4G_ECUDA;
}
