// bucket.cu — token -> expert bucketing for batched decode and chunked
// prefill (chenxutan ds4 article §2.3: router/expert fusion, chunked prefill).
// Integer work, bit-exact: counts, exclusive offsets, and a permutation that
// is stable in (t, k) order.  One CTA of 1024 threads walks the entries in
// chunks of 1024; inside a chunk, __match_any gives each entry its rank among
// equal experts of its warp, and per-warp counts in shared memory give the
// rank among earlier warps.
#include "ds4g_internal.cuh"

namespace ds4g {

__global__ void __launch_bounds__(1024) bucket_kernel(const int32_t *__restrict__ ids, int n,
                                                      int32_t *counts, int32_t *offsets,
                                                      int32_t *perm, int32_t *inv, uint32_t *status) {
    __shared__ int cnt[kE];
    __shared__ int base[kE];
    __shared__ int wc[32][kE];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < kE) cnt[tid] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += 1024) {
        const int e = ids[i];
        if ((unsigned)e < (unsigned)kE) atomicAdd(&cnt[e], 1);
        else flag_status(status, DS4G_EDEVICE, (uint32_t)e);
    }
    __syncthreads();
    if (warp == 0) {  // exclusive scan of 256 counts: 8 per lane
        int v[8], s = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[i] = cnt[8 * lane + i];
            s += v[i];
        }
        int incl = s;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        int run = incl - s;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            base[8 * lane + i] = run;
            counts[8 * lane + i] = v[i];
            offsets[8 * lane + i] = run;
            run += v[i];
        }
        if (lane == 31) offsets[kE] = run;
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    for (int c0 = 0; c0 < n; c0 += 1024) {
        for (int i = tid; i < 32 * kE; i += 1024) (&wc[0][0])[i] = 0;
        __syncthreads();
        const int i = c0 + tid;
        const int e = i < n ? ids[i] : -1;
        const bool valid = (unsigned)e < (unsigned)kE;
        const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : kE + lane);
        const int rank = __popc(peers & lt);
        if (valid && rank == 0) wc[warp][e] = __popc(peers);
        __syncthreads();
        if (valid) {
            int pre = 0;
            for (int w = 0; w < warp; ++w) pre += wc[w][e];
            const int pos = base[e] + pre + rank;
            perm[pos] = i;
            inv[i] = pos;
        } else if (i < n) {
            inv[i] = -1;
        }
        __syncthreads();
        if (tid < kE) {
            int s = 0;
            for (int w = 0; w < 32; ++w) s += wc[w][tid];
            base[tid] += s;
        }
        __syncthreads();
    }
}

}  // namespace ds4g

using namespace ds4g;

extern "C" size_t ds4g_bucket_workspace(int T) { return T < 1 ? 0 : kWsHeader; }

extern "C" ds4g_status ds4g_moe_bucket(const int32_t *ids, int T, int32_t *counts, int32_t *offsets,
                                       int32_t *perm, int32_t *inv, void *workspace, size_t ws_bytes,
                                       ds4g_stream_t s) {
    DS4G_TRACE();
    if (!ids || !counts || !offsets || !perm || !inv || !workspace || T < 1) return DS4G_EINVAL;
    if (((uintptr_t)ids | (uintptr_t)counts | (uintptr_t)offsets | (uintptr_t)perm | (uintptr_t)inv |
         (uintptr_t)workspace) & 15)
        return DS4G_EALIGN;
    if (ws_bytes < ds4g_bucket_workspace(T)) return DS4G_ENOSPACE;
    if ((long long)T * kK > (1ll << 30)) return DS4G_EUNSUPPORTED;
    bucket_kernel<<<1, 1024, 0, (cudaStream_t)s>>>(ids, T * kK, counts, offsets, perm, inv,
                                                    (uint32_t *)workspace);
    return cudaGetLastError() == cudaSuccess ? DS4G_OK : DS4G_ECUDA;
}

namespace ds4g {
// Launch helper for the prefill path (same kernel, status word given directly).
ds4g_status bucket_launch(const int32_t *ids, int T, int32_t *counts, int32_t *offsets, int32_t *perm,
                          int32_t *inv, uint32_t *status, cudaStream_t st) {
    bucket_kernel<<<1, 1024, 0, st>>>(ids, T * kK, counts, offsets, perm, inv, status);
    return cudaGetLastError() == cudaSuccess ? DS4G_OK : DS4G_ECUDA;
}
}  // namespace ds4g
