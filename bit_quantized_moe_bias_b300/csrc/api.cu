// api.cu — argument checks, workspace sizing and dispatch of the MoE block
// (chenxutan ds4 article §3.2 moe_forward), the RMS norm between chained
// layers (pages silent: eps 1e-6, no gain), and status reporting.
#include "ds4g_internal.cuh"

namespace ds4g {
size_t prefill_workspace(int T);
ds4g_status prefill_forward(const float *hidden, int T, const ds4g_layer *L, const int32_t *ids, const float *w,
                            float *out, void *workspace, cudaStream_t st, int phases);

// y = x / sqrt(mean(x^2) + 1e-6); one CTA of 256 threads per row of 4096.
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float *x, float *y) {
    const float4 *xr = reinterpret_cast<const float4 *>(x + (size_t)blockIdx.x * kH);
    float4 v[4];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[i] = xr[threadIdx.x + 256 * i];
        ss = fmaf(v[i].x, v[i].x, ss);
        ss = fmaf(v[i].y, v[i].y, ss);
        ss = fmaf(v[i].z, v[i].z, ss);
        ss = fmaf(v[i].w, v[i].w, ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    __shared__ float red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) tot += red[i];
    const float r = 1.0f / sqrtf(tot * (1.0f / kH) + 1e-6f);
    float4 *yr = reinterpret_cast<float4 *>(y + (size_t)blockIdx.x * kH);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        yr[threadIdx.x + 256 * i] = make_float4(v[i].x * r, v[i].y * r, v[i].z * r, v[i].w * r);
}

}  // namespace ds4g

using namespace ds4g;

extern "C" const char *ds4g_status_str(ds4g_status s) {
    switch (s) {
    case DS4G_OK: return "ok";
    case DS4G_EINVAL: return "invalid argument";
    case DS4G_EALIGN: return "device pointer not 16-byte aligned";
    case DS4G_ENOSPACE: return "workspace or buffer too small";
    case DS4G_ECUDA: return "CUDA error";
    case DS4G_EUNSUPPORTED: return "unsupported shape or type";
    case DS4G_ETIMEOUT: return "bounded device wait expired";
    case DS4G_EDEVICE: return "kernel flagged bad data";
    }
    return "unknown status";
}

// Bytes a call with exactly T tokens needs (the path T selects).
static size_t forward_ws_need(int T) {
    if (T < 1) return 0;
    if (T >= kPrefillMinT) return prefill_workspace(T);
    const size_t dec = decode_workspace(T < kDecodeMaxT ? T : kDecodeMaxT);
    if (T <= kDecodeMaxT) return dec;
    const size_t bat = batch_workspace(T);   // IQ2_XXS/Q2_K layers; Q4_K layers take the decode path
    return bat > dec ? bat : dec;
}

// The most any call with 1..T tokens needs: each path's need grows with T,
// so the maximum is over T and the largest T of every path below it.
extern "C" size_t ds4g_forward_workspace(int T) {
    if (T < 1) return 0;
    size_t n = forward_ws_need(T);
    const int tops[2] = {kDecodeMaxT, kPrefillMinT - 1};
    for (int i = 0; i < 2; ++i)
        if (tops[i] < T && forward_ws_need(tops[i]) > n) n = forward_ws_need(tops[i]);
    return n;
}

static bool types_ok(const ds4g_layer *L) {
    return (L->gate_up_type == DS4G_IQ2_XXS && L->down_type == DS4G_Q2_K) ||
           (L->gate_up_type == DS4G_Q4_K && L->down_type == DS4G_Q4_K);
}

static ds4g_status check_forward_args(const float *hidden, int T, const ds4g_layer *L,
                                      const int32_t *ids, const float *w, const float *out,
                                      const void *workspace, size_t ws_bytes) {
    if (!hidden || !L || !ids || !w || !out || !workspace || T < 1) return DS4G_EINVAL;
    if (!L->gate || !L->up || !L->down || !L->sh_gate || !L->sh_up || !L->sh_down) return DS4G_EINVAL;
    if (!types_ok(L)) return DS4G_EUNSUPPORTED;
    if (L->gate_up_type == DS4G_IQ2_XXS && !L->iq2_grid) return DS4G_EINVAL;
    const uintptr_t al = (uintptr_t)hidden | (uintptr_t)ids | (uintptr_t)w | (uintptr_t)out |
                         (uintptr_t)workspace | (uintptr_t)L->gate | (uintptr_t)L->up |
                         (uintptr_t)L->down | (uintptr_t)L->sh_gate | (uintptr_t)L->sh_up |
                         (uintptr_t)L->sh_down | (uintptr_t)L->iq2_grid;
    if (al & 15) return DS4G_EALIGN;
    if (ws_bytes < forward_ws_need(T)) return DS4G_ENOSPACE;
    return DS4G_OK;
}

static ds4g_status run_forward(const float *hidden, int T, const ds4g_layer *L, const int32_t *ids,
                               const float *w, float *out, void *workspace, size_t ws_bytes,
                               ds4g_stream_t s, int phases) {
    const ds4g_status chk = check_forward_args(hidden, T, L, ids, w, out, workspace, ws_bytes);
    if (chk != DS4G_OK) return chk;
    if (phases != 3 && T > kDecodeMaxT && T < kPrefillMinT) return DS4G_EUNSUPPORTED;
    cudaStream_t st = (cudaStream_t)s;
    if (T >= kPrefillMinT) {
        if ((long long)T * (kK + 1) * kH * 4 > (1ll << 40)) return DS4G_EUNSUPPORTED;
        return prefill_forward(hidden, T, L, ids, w, out, workspace, st, phases);
    }
    if (T > kDecodeMaxT && phases == 3 && L->gate_up_type == DS4G_IQ2_XXS)
        return batch_forward(hidden, T, L, ids, w, out, workspace, st);   // experts grouped: read once per chunk
    for (int t0 = 0; t0 < T; t0 += kDecodeMaxT) {
        const int n = T - t0 < kDecodeMaxT ? T - t0 : kDecodeMaxT;
        const ds4g_status rc = decode_forward(hidden + (size_t)t0 * kH, n, L, ids + (size_t)t0 * kK,
                                              w + (size_t)t0 * kK, out + (size_t)t0 * kH, workspace, st,
                                              phases);
        if (rc != DS4G_OK) return rc;
    }
    return DS4G_OK;
}

namespace ds4g {
ds4g_status forward_streamed_decode(const float *hidden, int T, const ds4g_layer *L, const int32_t *ids,
                                    const float *w, float *out, void *workspace, size_t ws_bytes, cudaStream_t st,
                                    const uint32_t *ready, uint32_t epoch) {
    const ds4g_status chk = check_forward_args(hidden, T, L, ids, w, out, workspace, ws_bytes);
    if (chk != DS4G_OK) return chk;
    if (T > kDecodeMaxT) return DS4G_EUNSUPPORTED;
    return decode_forward(hidden, T, L, ids, w, out, workspace, st, 3, nullptr, ready, epoch);
}
}  // namespace ds4g

extern "C" ds4g_status ds4g_moe_forward(const float *hidden, int T, const ds4g_layer *L,
                                        const int32_t *ids, const float *w, float *out,
                                        void *workspace, size_t ws_bytes, ds4g_stream_t s) {
    DS4G_TRACE();
    return run_forward(hidden, T, L, ids, w, out, workspace, ws_bytes, s, 3);
}

extern "C" ds4g_status ds4g_moe_forward_q8(const float *hidden, int T, const ds4g_layer *L,
                                           const int32_t *ids, const float *w, float *out,
                                           void *workspace, size_t ws_bytes, ds4g_stream_t s) {
    DS4G_TRACE();
    const ds4g_status chk = check_forward_args(hidden, T, L, ids, w, out, workspace, ws_bytes);
    if (chk != DS4G_OK) return chk;
    if (T > kDecodeMaxT || L->gate_up_type != DS4G_IQ2_XXS) return DS4G_EUNSUPPORTED;
    return decode_forward(hidden, T, L, ids, w, out, workspace, (cudaStream_t)s, 3, nullptr, nullptr, 0, 1);
}

extern "C" ds4g_status ds4g_moe_gate_up(const float *hidden, int T, const ds4g_layer *L,
                                        const int32_t *ids, const float *w, float *out,
                                        void *workspace, size_t ws_bytes, ds4g_stream_t s) {
    DS4G_TRACE();
    return run_forward(hidden, T, L, ids, w, out, workspace, ws_bytes, s, 1);
}

extern "C" ds4g_status ds4g_moe_down(const float *hidden, int T, const ds4g_layer *L,
                                     const int32_t *ids, const float *w, float *out,
                                     void *workspace, size_t ws_bytes, ds4g_stream_t s) {
    DS4G_TRACE();
    return run_forward(hidden, T, L, ids, w, out, workspace, ws_bytes, s, 2);
}

extern "C" ds4g_status ds4g_rmsnorm(const float *x, int T, float *y, ds4g_stream_t s) {
    DS4G_TRACE();
    if (!x || !y || T < 1) return DS4G_EINVAL;
    if (((uintptr_t)x | (uintptr_t)y) & 15) return DS4G_EALIGN;
    rmsnorm_kernel<<<T, 256, 0, (cudaStream_t)s>>>(x, y);
    return cudaGetLastError() == cudaSuccess ? DS4G_OK : DS4G_ECUDA;
}

extern "C" ds4g_status ds4g_last_error(void *workspace, ds4g_stream_t s) {
    if (!workspace) return DS4G_EINVAL;
    cudaStream_t st = (cudaStream_t)s;
    if (cudaStreamSynchronize(st) != cudaSuccess) return DS4G_ECUDA;
    uint32_t word[2] = {0, 0};
    if (cudaMemcpy(word, workspace, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return DS4G_ECUDA;
    if (word[0] != 0) {
        if (cudaMemset(workspace, 0, sizeof word) != cudaSuccess) return DS4G_ECUDA;
    }
    return (ds4g_status)word[0];
}
