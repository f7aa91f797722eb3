/*
 * ds4g.h — C ABI of the B300 routed-MoE block (libds4g.so).
 *
 * What it computes: the routed mixture-of-experts feed-forward block of
 * DeepSeek V4 Flash as the ds4 engine runs it with 2-bit experts:
 *   router scores -> top-6 of 256 experts -> for each selected expert a
 *   dequantise-inside-the-matmul SwiGLU MLP (gate/up IQ2_XXS, down Q2_K, or
 *   Q4_K for the q4 layers) -> weighted sum -> plus an always-on bf16 shared
 *   expert.
 *
 * Sources (web pages describing the ds4 engine):
 *   [P1] chenxutan.com, "ds4 深度实战：当 Redis 之父用纯 C 重写本地推理引擎":
 *        §2.1 (asymmetric 2-bit policy: gate/up IQ2_XXS, down Q2_K, shared
 *        expert and router kept at high precision), §2.3 (router+expert fusion,
 *        model-specific memory layout, chunked prefill), §3.2 (moe_forward:
 *        router -> only the routed experts -> shared expert -> merge).
 *   [P5] juejin.cn, "Redis 作者出手！ds4：用 C 语言从零打造 DeepSeek V4 Flash
 *        本地推理引擎": §2.1 (model constants: 4096 embd, 256 experts, 6 used,
 *        1 shared, 2048 expert FFN), §2.3 (block_q2_K 84 B and block_iq2_xxs
 *        66 B per 256 weights), §2.4 (the IQ2 grid-row dot kernel: a grid row is
 *        8 int8 values).
 * Where the pages are silent (score function, bias use, tie rule, inner bit
 * layout of the blocks, SwiGLU, RMS norm) the reading taken is stated at the
 * entry point that depends on it.
 *
 * Conventions (all entry points):
 *  - Dimensions are fixed: H = 4096 (hidden), F = 2048 (expert FFN),
 *    E = 256 experts, K = 6 used per token.  Other shapes -> DS4G_EUNSUPPORTED.
 *  - "dev" pointers are CUDA device pointers owned by the caller; "host"
 *    pointers are ordinary host memory owned by the caller.  The library never
 *    frees or retains a caller pointer beyond the call.
 *  - Every dev pointer must be 16-byte aligned, else DS4G_EALIGN.
 *  - All argument checks run on the host before any launch; a failed check
 *    launches nothing.  A failed launch returns DS4G_ECUDA.
 *  - GPU entry points are asynchronous on the given stream (0 = legacy
 *    default stream).  Faults the kernels detect (an expert id outside
 *    [0,256)) are recorded in a status word at the start of the workspace and
 *    read back by ds4g_last_error(); no kernel traps or spins unboundedly.
 *  - Hot entry points allocate nothing: scratch comes from the caller's
 *    workspace, sized by the matching *_workspace() query.
 *  - Row-major everywhere: hidden[T][4096]; a weight matrix [rows][cols] has
 *    rows = output features, cols = input features.
 *  - One GPU per process: kernel attributes (dynamic shared memory) and the
 *    SM count that sizes the persistent grids are set up on first use, for
 *    the device current at that time.  Driving several GPUs from one process
 *    is not supported; run one process per GPU.
 */
#ifndef DS4G_H
#define DS4G_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *ds4g_stream_t; /* == cudaStream_t */

#define DS4G_N_EMBD        4096
#define DS4G_N_FF_EXP      2048
#define DS4G_N_EXPERT      256
#define DS4G_N_EXPERT_USED 6

typedef enum {
    DS4G_OK = 0,
    DS4G_EINVAL = 1,       /* NULL pointer, T < 1, bad enum, inconsistent sizes */
    DS4G_EALIGN = 2,       /* a device pointer is not 16-byte aligned          */
    DS4G_ENOSPACE = 3,     /* workspace or output buffer too small             */
    DS4G_ECUDA = 4,        /* a CUDA runtime call or launch failed             */
    DS4G_EUNSUPPORTED = 5, /* shape or type combination not implemented        */
    DS4G_ETIMEOUT = 6,     /* a bounded device wait gave up                    */
    DS4G_EDEVICE = 7       /* a kernel flagged bad data (e.g. expert id >= 256)*/
} ds4g_status;

typedef enum {
    DS4G_IQ2_XXS = 0, /* 66 B / 256 weights: fp16 d, 64 B of grid/sign codes  */
    DS4G_Q2_K = 1,    /* 84 B / 256: scales[16], qs[64], fp16 d, fp16 dmin    */
    DS4G_Q4_K = 2,    /* 144 B / 256: fp16 d, fp16 dmin, scales[12], qs[128]  */
    DS4G_BF16 = 3     /* plain bf16, 2 B / weight                              */
} ds4g_qtype;

/* Human-readable name of a status code (static string, never NULL). */
const char *ds4g_status_str(ds4g_status s);

/* ------------------------------------------------------------------------
 * Block formats and the device layout ("model-specific memory layout",
 * [P1] §2.3).  The GGUF-format blocks are the structs of [P5] §2.3 laid end to
 * end, row by row (row r, block b at byte (r*cols/256 + b)*block_bytes).
 * The device ("packed") layout is a pure byte/bit permutation of the same
 * content into 16-row tiles so that each GPU lane reads exactly the codes it
 * multiplies; it holds the same number of bytes.  No arithmetic is done.
 * ------------------------------------------------------------------------ */

/* Bytes of one 256-weight block in GGUF format (66, 84, 144; 512 for BF16). */
size_t ds4g_block_bytes(ds4g_qtype t);

/* Bytes of a packed [rows][cols] matrix (== GGUF bytes).  0 if the shape is
 * invalid (rows % 16 != 0 or cols % 256 != 0) or t is DS4G_BF16. */
size_t ds4g_packed_size(ds4g_qtype t, int rows, int cols);

/* Host-only.  GGUF-format blocks (host, in_bytes) -> packed layout (host,
 * out_bytes).  Layout only.  Errors: EINVAL (NULL, bad type), EUNSUPPORTED
 * (shape), ENOSPACE (in_bytes or out_bytes below ds4g_packed_size). */
ds4g_status ds4g_quantize_pack(ds4g_qtype t, int rows, int cols,
                               const void *gguf_blocks, size_t in_bytes,
                               void *packed, size_t out_bytes);

/* Host-only inverse of ds4g_quantize_pack (used by tests: round trip). */
ds4g_status ds4g_unpack(ds4g_qtype t, int rows, int cols,
                        const void *packed, size_t in_bytes,
                        void *gguf_blocks, size_t out_bytes);

/* Device twin of ds4g_quantize_pack for resident model loading: gguf_dev and
 * packed_dev are device buffers of ds4g_packed_size() bytes (must not
 * overlap).  Asynchronous on stream s.  Same errors as the host version plus
 * EALIGN / ECUDA. */
ds4g_status ds4g_quantize_pack_device(ds4g_qtype t, int rows, int cols,
                                      const void *gguf_dev, void *packed_dev,
                                      ds4g_stream_t s);

/* Dequantise a packed matrix to fp32 and/or bf16 (bf16 = round-to-nearest-
 * even of the fp32 value).  Exposes the arithmetic the MoE kernels use so it
 * can be checked bit for bit:
 *   IQ2_XXS: w = ((d * (0.5 + ls)) * 0.25) * (+-grid[a][j])       ([P5] §2.3)
 *   Q2_K/Q4_K: w = fma(d * sc, q, -(dmin * m))
 * each step one IEEE fp32 rounding.  iq2_grid (dev, 256 x 8 int8 packed as
 * uint64, little-endian bytes) is required for IQ2_XXS, ignored otherwise.
 * out_f32 [rows][cols] and out_bf16 [rows][cols] (bf16 bits) are dev; either
 * may be NULL but not both. */
ds4g_status ds4g_dequantize(ds4g_qtype t, const void *packed, int rows, int cols,
                            const uint64_t *iq2_grid, float *out_f32,
                            uint16_t *out_bf16, ds4g_stream_t s);

/* ------------------------------------------------------------------------
 * Router ([P1] §3.2 "Router 计算专家选择"; [P5] §2.1 DS4_N_EXPERT_USED = 6).
 * For each token t (reading for what the pages leave open: sigmoid scores,
 * bias used only to select, ties to the lower expert id, weights = selected
 * unbiased scores renormalised to sum 1, no extra scale factor):
 *   logit_e = sum_j hidden[t][j] * router[e][j]       (fp32 accumulate)
 *   s_e     = 1 / (1 + exp(-logit_e))
 *   ids[t]  = the 6 experts with the largest s_e + bias[e], largest first,
 *             equal keys -> lower e first
 *   w[t][k] = s_{ids[t][k]} / sum_k' s_{ids[t][k']}
 * hidden [T][4096] f32 dev, router [256][4096] f32 dev, bias [256] f32 dev,
 * ids [T][6] int32 dev, w [T][6] f32 dev, workspace dev of at least
 * ds4g_route_workspace(T) bytes (the status word, ticket counters and the
 * logits), zeroed once before first use: the kernels leave the counters at
 * zero, and they sit at the same offsets for every T, so one workspace
 * serves calls with any T it is large enough for.  ds4g_route_workspace(T)
 * is the most that any call with 1..T tokens needs (non-decreasing in T), so
 * a workspace sized for the largest T serves every smaller call.
 * 1 <= T <= DS4G_ROUTE_MAX_T, else DS4G_EINVAL / DS4G_EUNSUPPORTED
 * (ds4g_route_workspace returns 0 outside that range).
 * ------------------------------------------------------------------------ */
#define DS4G_ROUTE_MAX_T (1 << 20)
size_t ds4g_route_workspace(int T);
ds4g_status ds4g_moe_route(const float *hidden, int T, const float *router,
                           const float *bias, int32_t *ids, float *w,
                           void *workspace, size_t ws_bytes, ds4g_stream_t s);

/* ------------------------------------------------------------------------
 * Token -> expert bucketing (batched decode and chunked prefill, [P1] §2.3).
 * For the 6T entries (t,k) in row-major order:
 *   counts[e]   = number of entries with ids[t][k] == e          (e < 256)
 *   offsets[e]  = sum_{e' < e} counts[e'];  offsets[256] = 6T
 *   perm[offsets[e] + r] = t*6 + k of the r-th entry (in (t,k) order) of e
 *   inv[t*6 + k] = its position in perm  (perm[inv[i]] == i)
 * Integer work, bit-exact.  All arrays dev int32.  An id outside [0,256)
 * sets DS4G_EDEVICE in the workspace status word and is counted nowhere.
 * ------------------------------------------------------------------------ */
size_t ds4g_bucket_workspace(int T);
ds4g_status ds4g_moe_bucket(const int32_t *ids, int T, int32_t *counts,
                            int32_t *offsets, int32_t *perm, int32_t *inv,
                            void *workspace, size_t ws_bytes, ds4g_stream_t s);

/* ------------------------------------------------------------------------
 * One MoE layer's weights, all device memory owned by the caller.
 * gate/up/down are device arrays of 256 device pointers, one packed matrix
 * per expert: gate/up [2048][4096] of gate_up_type, down [4096][2048] of
 * down_type.  Supported pairs: (IQ2_XXS, Q2_K) — the q2 layers — and
 * (Q4_K, Q4_K) — the q4 layers of the q2-q4 model ([P1] §2.1).
 * Shared expert: bf16 bits, row-major, sh_gate/sh_up [2048][4096],
 * sh_down [4096][2048] (kept unquantised, [P1] §2.1).
 * iq2_grid: 256 rows of 8 int8 grid values (IQ2_XXS codebook), dev.
 * ------------------------------------------------------------------------ */
typedef struct {
    ds4g_qtype gate_up_type;
    ds4g_qtype down_type;
    const void *const *gate;
    const void *const *up;
    const void *const *down;
    const uint16_t *sh_gate;
    const uint16_t *sh_up;
    const uint16_t *sh_down;
    const uint64_t *iq2_grid;
} ds4g_layer;

/* ------------------------------------------------------------------------
 * The MoE block given the routing ([P1] §3.2 moe_forward).  For each token t:
 *   for k in 0..5, e = ids[t][k]:
 *     g = G_e x, u = U_e x  (weights dequantised inside the matmul)
 *     h_k = silu(g) * u                        (SwiGLU, no clamp)
 *     y_k = D_e h_k
 *   s = Sd (silu(Sg x) * (Su x))                (bf16 shared expert)
 *   out[t] = s + sum_{k=0..5} w[t][k] * y_k     (fixed k order, no atomics)
 * hidden [T][4096] f32 dev, ids [T][6] int32 dev, w [T][6] f32 dev,
 * out [T][4096] f32 dev.  A repeated id within a token is legal (both terms
 * are summed).  Three paths, chosen by T:
 *  - T <= 3, and Q4_K layers up to T = 63 (decode): per-slot
 *    dequant-in-register GEMV, processed in chunks of 3 tokens.  Codes enter
 *    the tensor cores exactly; activations as an fp16 hi+lo pair
 *    (|x| < 65504 required, else DS4G_EDEVICE); h as an fp16 hi+lo pair
 *    scaled by a power of two per 16 entries (any finite h; inf/NaN is
 *    DS4G_EDEVICE); fp32 accumulation.  Expected error ~1e-5 relative.
 *  - 4 <= T < 64 with IQ2_XXS/Q2_K layers (batched decode): the slots
 *    grouped by expert, each selected expert's weights read once per chunk
 *    of up to 32 tokens and applied to all of its tokens.  Same arithmetic as
 *    the per-slot path except that h enters the down projection as fp16 of
 *    2^-e h without a lo part, and the shared expert's bf16 weights as fp16.
 *    Expected error ~1e-4 relative.
 *  - T >= 64 (chunked prefill, large batches): tokens bucketed by expert,
 *    grouped tcgen05 GEMM.  Routed weights are the fp32 block formula
 *    rounded to nearest even in fp16, against fp16 activations (gate/up;
 *    |x| < 65504 required, else DS4G_EDEVICE) and fp16 h scaled by a power
 *    of two per row (down); bf16 throughout for the shared expert; fp32
 *    accumulation.  Expected error ~1e-3 relative L2 per token.
 * workspace dev >= ds4g_forward_workspace(T) bytes (about 200 KB per token
 * on the prefill path), zeroed once before first use; one call at a time.
 * Workspace reuse: every workspace of this family (ds4g_moe_forward,
 * ds4g_moe_layer_decode, ds4g_moe_decode_stack) keeps its kernels' counters
 * in one area at fixed offsets after the status word, which every kernel
 * leaves at zero and no call uses as scratch; so one workspace, large enough
 * for each call, serves any sequence of these calls and token counts.
 * ds4g_forward_workspace(T) is the most that any call with 1..T tokens needs
 * (non-decreasing in T, across the three paths), so a workspace sized for the
 * largest T serves every smaller call.
 * ------------------------------------------------------------------------ */
size_t ds4g_forward_workspace(int T);
ds4g_status ds4g_moe_forward(const float *hidden, int T, const ds4g_layer *L,
                             const int32_t *ids, const float *w, float *out,
                             void *workspace, size_t ws_bytes, ds4g_stream_t s);

/* The two phases of ds4g_moe_forward, for callers that schedule them
 * separately (e.g. to overlap other work between them, or to time them):
 * ds4g_moe_gate_up computes h_k = silu(G_e x) * (U_e x) for every slot and
 * the shared expert into the workspace; ds4g_moe_down reads them from the
 * same workspace and writes out.  Same arguments and checks as
 * ds4g_moe_forward; calling gate_up then down on the same workspace and
 * stream equals one ds4g_moe_forward.  For T <= 3 (one decode chunk) or
 * T >= 64 (prefill path: gate_up = bucketing, permute and the gate/up GEMM;
 * down = the down GEMM and the combine); other T -> DS4G_EUNSUPPORTED. */
ds4g_status ds4g_moe_gate_up(const float *hidden, int T, const ds4g_layer *L,
                             const int32_t *ids, const float *w, float *out,
                             void *workspace, size_t ws_bytes, ds4g_stream_t s);
ds4g_status ds4g_moe_down(const float *hidden, int T, const ds4g_layer *L,
                          const int32_t *ids, const float *w, float *out,
                          void *workspace, size_t ws_bytes, ds4g_stream_t s);

/* ------------------------------------------------------------------------
 * The int8-activation decode path (chenxutan ds4 article §2.4: the
 * dot_iq2_pair_16 kernel, int8 grid values against int8 activations; here
 * with dp4a).  ds4g_moe_forward for 1 <= T <= 3 with the routed IQ2_XXS gate
 * and up projections on q8 activations: per token and 256-column block,
 * d = max|x| / 127 (fp32) and q = x / d rounded to nearest, ties to even,
 * clamped to +-127 (a reading: the pages give the dot, not the quantiser);
 * per 32-weight sub-block the exact integer sum S of (sign * grid value) * q,
 * then d_sub * d * S in fp32.  The down projection, the shared expert and
 * everything else are those of ds4g_moe_forward.  Same arguments and checks;
 * T > 3 or a gate/up type other than IQ2_XXS: DS4G_EUNSUPPORTED.  Results
 * differ from ds4g_moe_forward by the activation rounding (about 0.4 % of
 * each block's largest value per entry): an alternative path, not the
 * default (see the design notes for its measured speed).
 * ------------------------------------------------------------------------ */
ds4g_status ds4g_moe_forward_q8(const float *hidden, int T, const ds4g_layer *L,
                                const int32_t *ids, const float *w, float *out,
                                void *workspace, size_t ws_bytes, ds4g_stream_t s);

/* ------------------------------------------------------------------------
 * One decode token through one whole MoE layer in a single launch ([P1]
 * §2.3: router logic and expert compute fused into one GPU dispatch; §3.2
 * moe_forward).  With xn = hidden / sqrt(mean(hidden^2) + 1e-6) if normalize
 * is non-zero, else xn = hidden:
 *   ids, w = the router of ds4g_moe_route applied to xn
 *   out    = ds4g_moe_forward(xn, ids, w)
 * hidden [4096] f32 dev (T = 1), router [256][4096] f32 dev, bias [256] f32
 * dev, ids [6] int32 dev (out), w [6] f32 dev (out), out [4096] f32 dev.
 * Layer types: IQ2_XXS gate/up with Q2_K down, or Q4_K gate/up/down (the q4
 * layers of the q2-q4 model, [P1] §2.1; iq2_grid may be NULL for them); any
 * other pair -> DS4G_EUNSUPPORTED.  Arithmetic as the decode path of
 * ds4g_moe_forward (exact codes, fp16 hi+lo activation, fp32 scales), except
 * that the shared expert runs on bf16 tensor cores with the activation and
 * the shared h as bf16 hi+lo pairs.  workspace dev >= ds4g_layer_decode_workspace()
 * bytes, zeroed once before first use (the kernel leaves its counters at
 * zero); one call at a time per workspace.  h enters the down projection
 * as an fp16 hi+lo pair scaled by a power of two per 16 entries (any finite
 * h).  Kernel-detected faults (bad expert id, |xn| >= 65504, a non-finite h,
 * a bounded wait that expired) are read
 * back with ds4g_last_error(workspace); so is an IQ2_XXS grid byte outside
 * {8, 25, 43}, the format's magnitudes (DS4G_EUNSUPPORTED: this kernel
 * encodes grid rows as 2-bit codes of those values).
 * The kernel keeps one CTA on every SM and its CTAs wait on each other
 * (bounded), so it needs the whole GPU: run nothing else concurrently.  The
 * first call checks that one CTA (its threads and 227 KB of shared memory)
 * fits on an SM, and returns DS4G_EUNSUPPORTED without launching if not; a
 * kernel of another stream or process that holds SMs for longer than the
 * bounded waits (about 1 s) makes the call end with DS4G_ETIMEOUT, read
 * back with ds4g_last_error.
 * ------------------------------------------------------------------------ */
size_t ds4g_layer_decode_workspace(void);
ds4g_status ds4g_moe_layer_decode(const float *hidden, int normalize, const float *router,
                                  const float *bias, const ds4g_layer *L, int32_t *ids,
                                  float *w, float *out, void *workspace, size_t ws_bytes,
                                  ds4g_stream_t s);

/* ------------------------------------------------------------------------
 * One decode token through n_layers chained MoE layers on the input
 *   x_0 = hidden,  x_l = output of layer l-1  (l >= 1);
 * every layer's input is RMS-normalised and no residual is added (the
 * full-depth decode workload of 43 such layers).  Layer l is
 * ds4g_moe_layer_decode with normalize = 1, for either layer type that call
 * takes (IQ2_XXS/Q2_K, or Q4_K throughout: the q2-q4 and q4 models,
 * chenxutan ds4 article §2.1); any other type pair: DS4G_EUNSUPPORTED.
 *   hidden   [4096] f32 dev            routers  host array [n_layers] of dev
 *   layers   host array [n_layers]       pointers to [256][4096] f32
 *   biases   host array [n_layers] of dev pointers to [256] f32
 *   ids      [n_layers][6] int32 dev (out)   w  [n_layers][6] f32 dev (out)
 *   hbuf     [2][4096] f32 dev: scratch for the intermediate outputs
 *   out      [4096] f32 dev: the last layer's output
 *   workspace dev, zeroed once before first use, one call at a time; one
 *            workspace serves all layers: >= ds4g_decode_stack_workspace()
 *            bytes (equal to ds4g_layer_decode_workspace()), else
 *            DS4G_ENOSPACE.  Faults are read with ds4g_last_error.
 * 1 <= n_layers <= 1024, else DS4G_EINVAL.  All checks of every layer run
 * before the first launch.  Same results, bit for bit, as the per-layer
 * calls.  Every layer after the first is a programmatic dependent launch of
 * the previous one: its CTAs start on the SMs that the previous
 * layer's CTAs leave, build their tables and begin streaming the layer's
 * router and shared-expert weights, and read their input and the workspace
 * only after the previous layer has completed.
 * ------------------------------------------------------------------------ */
size_t ds4g_decode_stack_workspace(void);
ds4g_status ds4g_moe_decode_stack(const float *hidden, int n_layers, const float *const *routers,
                                  const float *const *biases, const ds4g_layer *layers,
                                  int32_t *ids, float *w, float *hbuf, float *out,
                                  void *workspace, size_t ws_bytes, ds4g_stream_t s);

/* ------------------------------------------------------------------------
 * Test hook of the bounded waits (no counterpart in the pages: it exists to
 * exercise DS4G_ETIMEOUT without hanging or faulting a GPU).  While on != 0,
 * every launch of the fused layer kernel (ds4g_moe_layer_decode and every
 * layer of ds4g_moe_decode_stack) makes its control warps wait
 * for one router row more than the layer has, giving up after about 130 us:
 * the launch aborts, drains its copies, records DS4G_ETIMEOUT in the
 * workspace and leaves it usable.  Process-wide, host-side only;
 * turn it off (0) to run normally.  Not for production use.
 * ------------------------------------------------------------------------ */
void ds4g_test_force_timeout(int on);

/* ------------------------------------------------------------------------
 * ds4g_moe_forward without a workspace, for callers that cannot allocate
 * device memory: code running inside an allocator or memory-pool callback
 * (where calling cudaMalloc would re-enter the allocator), a real-time loop
 * that must never stall on the driver's allocator, or a plugin whose host
 * engine hands it fixed input/output buffers and owns all other memory.
 * (The ds4 pages have no counterpart: their engine owns all its memory.)
 *
 * Arguments and checks are those of ds4g_moe_forward minus the workspace;
 * the caller still passes hidden, ids, w and out.  Whatever T, the call runs
 * the per-slot decode kernels of ds4g_moe_forward on chunks of up to three
 * tokens, so it returns, bit for bit, what ds4g_moe_forward returns when
 * called on the same chunks one at a time.  For a whole batch of T >= 4
 * tokens ds4g_moe_forward takes other kernels (the batched path from T = 4
 * for IQ2_XXS/Q2_K layers, the tensor-core prefill path from T = 64): their
 * results agree with this
 * call within the block's tolerance, not bit for bit, and they read each
 * selected expert's weights once per batch, where this call reads them once
 * per chunk.  Scratch is a library-owned device array of 5 MB (file scope,
 * one per device that loads the library, held until the process exits).
 * Limits and behaviour:
 *  - 1 <= T <= DS4G_NOALLOC_MAX_T, else DS4G_EINVAL (T < 1) or
 *    DS4G_ENOSPACE (T too large), returned before any CUDA call.
 *  - Allocates nothing: no cudaMalloc/cudaFree and no allocating library
 *    call.  Every call clears the array's status word and tile counters
 *    (13 KB) with cudaMemsetAsync on s, then runs the decode kernels on s.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current and keeps it for the
 *    process; make that first call before any stream capture.  After a
 *    cudaDeviceReset the kept address is stale: the call is not supported
 *    on a device that has been reset.
 *  - All calls share the one array: calls that overlap on the GPU (other
 *    streams, other host threads) race and give wrong results.  Serialise
 *    them, e.g. on one stream.
 *  - Faults the kernels detect (a bad expert id) are recorded in the array's
 *    status word, which no entry point reads back; callers that need that
 *    check use ds4g_moe_forward with a workspace and ds4g_last_error.
 * ------------------------------------------------------------------------ */
#define DS4G_NOALLOC_MAX_T 64
ds4g_status ds4g_moe_forward_noalloc(const float *hidden, int T, const ds4g_layer *L,
                                     const int32_t *ids, const float *w, float *out,
                                     ds4g_stream_t s);

/* ------------------------------------------------------------------------
 * Expert streaming: routed experts held in host memory, an HBM expert cache.
 * [P1] §3.3 (routed experts loaded as the router selects them), §3.5 "SSD
 * streaming", and the yudady DS-4 DwarfStar page, section
 * "SSD Streaming": when the model does not fit the GPU's memory, the
 * non-routed weights stay resident and a routed expert that misses the cache
 * is loaded, used, and its space later released.  Here the routed experts of
 * any number of layers live in host memory; a device pool of n_slots expert
 * slots (gate + up + down of one expert each) keeps the most recently used
 * ones, evicting the least recently used slot that the current call does not
 * need; a slot is keyed by (layer_key, expert).
 *
 * ds4g_expert_cache_pool_bytes: device bytes of the pool for n_slots slots
 *   of the type pair (the slots, a 6 KB pointer table and 256 B of ready
 *   flags); 0 for an
 *   unsupported pair or n_slots < 1.
 * ds4g_expert_cache_create: pool dev, 16-byte aligned, >= pool_bytes, owned
 *   by the caller and kept alive until destroy.  The cache object and two
 *   small pinned host staging buffers are allocated here (create/destroy are
 *   not hot calls).  max_tokens bounds T of the forwards.  Errors:
 *   DS4G_EINVAL (NULL argument, n_slots < 6, max_tokens < 1 or > 2^20),
 *   DS4G_EUNSUPPORTED (type pair), DS4G_EALIGN, DS4G_ENOSPACE (pool too
 *   small), DS4G_ECUDA (staging allocation failed).
 * ds4g_expert_cache_destroy: frees what create allocated (not the pool); no
 *   forward using the cache may be in flight.
 * ds4g_expert_cache_stats: since create, the distinct experts per call that
 *   were resident (hits) or copied in (misses), and the bytes copied.
 *
 * ds4g_moe_forward_streamed: ds4g_moe_forward for T tokens of one layer whose
 * routed experts come from host memory.
 *   src->gate/up/down: host arrays [256] of host pointers to each expert's
 *     packed matrices (layout of ds4g_quantize_pack; pinned memory, e.g. from
 *     cudaHostAlloc, so that the copies are asynchronous); NULL for an expert
 *     the caller does not provide.  Types must equal the cache's.
 *   layer_key >= 0 names the layer in the cache's keys.
 *   sh_*, iq2_grid (dev), hidden, ids, w, out, workspace as for
 *     ds4g_moe_forward.
 * Steps: copy ids to the host and synchronise s (this also retires the
 * kernels and copies of every earlier call on the cache, so any slot may be
 * rewritten); give each distinct selected expert its slot; copy the pointer
 * tables on s; copy the experts not resident (three cudaMemcpyAsync each).
 * For T <= 3 the copies run on the cache's own copy stream while the decode
 * kernels of ds4g_moe_forward already run on s: the shared expert's work
 * first, and each slot's routed work once a flag, written on the copy stream
 * after that slot's expert, shows it has landed (a bounded wait; s then
 * waits for the copies).  For larger T the copies come first on s, then
 * ds4g_moe_forward.
 * Output bit-identical to ds4g_moe_forward with the same experts resident.
 * Errors: T < 1 or > max_tokens, NULL argument, a selected expert whose host
 * pointer is NULL: DS4G_EINVAL; more distinct experts than n_slots:
 * DS4G_ENOSPACE; types differing from the cache's: DS4G_EUNSUPPORTED; then
 * the errors of ds4g_moe_forward.  An id outside [0,256) is left to the
 * kernels (DS4G_EDEVICE in the workspace).  The host blocks until s drains:
 * use one stream for all calls on a cache.
 *
 * ds4g_expert_lru_simulate (exported for tests; no GPU): runs the cache's
 * slot policy over n_calls calls of call_sizes[c] keys each (keys host
 * int64, concatenated; < 0 = skipped) on n_slots empty slots and writes, per
 * key, its slot (-1 for a skipped key) and 1 if it would be copied in; a
 * call with more distinct keys than slots gets slot -2 for all its keys
 * (the forward's DS4G_ENOSPACE) and the next call proceeds.
 * ------------------------------------------------------------------------ */
typedef struct ds4g_expert_cache ds4g_expert_cache;
typedef struct {
    ds4g_qtype gate_up_type;
    ds4g_qtype down_type;
    const void *const *gate;   /* host [256] of host pointers */
    const void *const *up;
    const void *const *down;
} ds4g_host_experts;
size_t ds4g_expert_cache_pool_bytes(ds4g_qtype gate_up_type, ds4g_qtype down_type, int n_slots);
ds4g_status ds4g_expert_cache_create(ds4g_qtype gate_up_type, ds4g_qtype down_type, int n_slots,
                                     int max_tokens, void *pool, size_t pool_bytes,
                                     ds4g_expert_cache **cache);
ds4g_status ds4g_expert_cache_destroy(ds4g_expert_cache *cache);
ds4g_status ds4g_expert_cache_stats(const ds4g_expert_cache *cache, uint64_t *hits,
                                    uint64_t *misses, uint64_t *bytes_copied);
ds4g_status ds4g_moe_forward_streamed(const float *hidden, int T, int layer_key,
                                      const ds4g_host_experts *src, const uint16_t *sh_gate,
                                      const uint16_t *sh_up, const uint16_t *sh_down,
                                      const uint64_t *iq2_grid, const int32_t *ids,
                                      const float *w, float *out, ds4g_expert_cache *cache,
                                      void *workspace, size_t ws_bytes, ds4g_stream_t s);
ds4g_status ds4g_expert_lru_simulate(int n_slots, int n_calls, const int32_t *call_sizes,
                                     const int64_t *keys, int32_t *slot_out, uint8_t *miss_out);

/* ------------------------------------------------------------------------
 * Expert files: the routed experts of one layer read from storage when they
 * miss the cache ([P1] §3.5 "SSD streaming"; the yudady DS-4 DwarfStar page,
 * "SSD Streaming").  File layout (little-endian): a 4096-byte header —
 * magic "DS4GEXP1", uint32 gate_up_type, uint32 down_type, uint32 256,
 * uint32 0, uint64 bytes of one packed gate (= up) matrix, uint64 bytes of
 * one packed down matrix, uint64 record stride, a 32-byte presence bitmap
 * (bit e % 8 of byte e / 8: expert e stored), zeros — then expert e's packed
 * gate, up and down (the layout of ds4g_quantize_pack) back to back at byte
 * 4096 + e * stride; stride = that record's size rounded up to 4096.
 *
 * ds4g_expert_file_write: writes src's experts (host pointers; an expert
 *   whose three pointers are NULL is not stored, and a partial one is
 *   DS4G_EINVAL) to path, replacing the file.  No CUDA call.  Errors:
 *   DS4G_EINVAL (NULL argument, partial expert, I/O failure),
 *   DS4G_EUNSUPPORTED (type pair).
 * ds4g_expert_file_open: validates the header (magic, types, sizes, stride,
 *   file length; DS4G_EINVAL before any CUDA call if one is wrong) and
 *   allocates two pinned staging buffers of one expert each; the handle
 *   keeps the file open.  ds4g_expert_file_close waits for the staging
 *   buffers' last copies, frees them and closes the file.
 * ds4g_moe_forward_streamed_file: ds4g_moe_forward_streamed with the missing
 *   experts read from the file: each is read (pread) into a staging buffer
 *   and copied to its slot on s; the read of one expert overlaps the copy
 *   of the one before (a buffer is reused after its copy's event).  Same
 *   results, bit for bit, and the same errors; an expert absent from the
 *   file, or a failed read, is DS4G_EINVAL.  The cache's types must equal
 *   the file's.  One call at a time per file handle.
 * ------------------------------------------------------------------------ */
typedef struct ds4g_expert_file ds4g_expert_file;
ds4g_status ds4g_expert_file_write(const char *path, const ds4g_host_experts *src);
ds4g_status ds4g_expert_file_open(const char *path, ds4g_expert_file **file);
ds4g_status ds4g_expert_file_close(ds4g_expert_file *file);
ds4g_status ds4g_moe_forward_streamed_file(const float *hidden, int T, int layer_key,
                                           ds4g_expert_file *file, const uint16_t *sh_gate,
                                           const uint16_t *sh_up, const uint16_t *sh_down,
                                           const uint64_t *iq2_grid, const int32_t *ids,
                                           const float *w, float *out, ds4g_expert_cache *cache,
                                           void *workspace, size_t ws_bytes, ds4g_stream_t s);

/* RMS norm between chained layers (pages silent; reading: eps = 1e-6, no
 * learned gain): y[t] = x[t] / sqrt(mean_j x[t][j]^2 + 1e-6).  In place
 * (x == y) is allowed.  x, y [T][4096] f32 dev. */
ds4g_status ds4g_rmsnorm(const float *x, int T, float *y, ds4g_stream_t s);

/* Synchronises stream s, reads the status word in workspace (dev) and
 * returns it (DS4G_OK if no kernel flagged anything), then clears it. */
ds4g_status ds4g_last_error(void *workspace, ds4g_stream_t s);

#ifdef __cplusplus
}
#endif
#endif /* DS4G_H */
