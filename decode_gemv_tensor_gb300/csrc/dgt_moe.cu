// dgt_moe.cu -- mixture-of-experts expert-gather products with R4 (or BF16)
// expert weights, in the batch-1 product's fixed summation order.
//
// Binade README, "How it works" (Exactness: "the matvec, the MoE expert
// gather and the GEMM" follow one order) and "Limitations" (the fused kernels
// cover "every expert product").  The experts of one projection are stacked
// as one tensor [E * Ne, K] with one rank table.  For token t and slot j,
// y[t, j, :] = W[ids[t, j]] x_t in the order of dgt_gemv (plan S(Ne, K));
// with routing weights p, out[t, :] = fmaf chain over j = 0..topk-1 of
// p[t, j] * y[t, j, :], starting from +0.
//
// Three launches:
//  1. k_moe_route (one CTA): counts the pairs per expert, lists the experts
//     in use, and places every pair (t, j) in its expert's list in (t, j)
//     order -- deterministic, no atomics in the placement.
//  2. k_moe: a warp takes two rows of an expert in use at a time and streams
//     each row once (up to 8 rounds of loads in flight), decodes each 16-weight
//     lane chunk once and runs one fmaf chain per routed token (up to 4 per
//     pass) against x staged in shared memory; at each slice end the chains
//     are butterfly-reduced into the workspace.
//  3. k_moe_combine: adds each pair's slices left to right (y) and applies
//     the routing weights in slot order (out).
#include <cuda_runtime.h>

#include "../../include/dgt.h"
#include "dgt_device.cuh"
#include "dgt_internal.h"
#include "dgt_launch.h"

namespace dgt {

constexpr int MW = 8;               // warps per CTA
constexpr uint32_t MOE_TPASS = 4;   // tokens per pass over a row
constexpr uint32_t MOE_MAX_EXPERTS = 4096;
constexpr uint32_t MOE_MAX_PAIRS = 1u << 16;
constexpr uint32_t MOE_XS_LIMIT = 160 * 1024;  // x of every token in shared memory

struct MoeArgs {
    const uint8_t *sm, *nib, *esc;
    const uint32_t *seg;
    const uint16_t *W;
    const int32_t *ids;
    const float *p;
    const uint16_t *x;
    float *y32;
    uint16_t *out;
    float *out32;
    uint64_t cols, nseg, n_esc, ne;
    uint32_t n_experts, tokens, topk, J, S;
    R4Lut L;
    uint8_t table[256];
    // workspace
    uint32_t *eoff;    // n_experts + 1
    uint32_t *elist;   // pairs: t << 8 | j
    uint32_t *active;  // experts in use, then the count at active[pairs]
    float *partial;    // pairs * ne * S
    int32_t *status;
};

static inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct WsLayout {
    size_t eoff, elist, active, partial, total;
};

static inline WsLayout moe_ws_layout(uint32_t n_experts, uint64_t ne, uint64_t cols, uint32_t tokens,
                                     uint32_t topk) {
    const uint64_t pairs = (uint64_t)tokens * topk;
    const int S = dgt_plan_slices(ne, cols);
    WsLayout l;
    l.eoff = 0;
    l.elist = align256(l.eoff + 4ull * (n_experts + 1));
    l.active = align256(l.elist + 4ull * pairs);
    l.partial = align256(l.active + 4ull * (pairs + 1));
    l.total = align256(l.partial + 4ull * pairs * ne * (uint64_t)S);
    return l;
}

__global__ void __launch_bounds__(1024) k_moe_route(MoeArgs a) {
    __shared__ uint32_t cnt[MOE_MAX_EXPERTS];
    __shared__ uint32_t nact;
    const uint32_t P = a.tokens * a.topk;
    for (uint32_t e = threadIdx.x; e < a.n_experts; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    for (uint32_t q = threadIdx.x; q < P; q += blockDim.x) {
        const int32_t e = a.ids[q];
        if (e < 0 || (uint32_t)e >= a.n_experts) {
            set_status(a.status, DGT_ERR_ARG);
            continue;
        }
        atomicAdd(&cnt[e], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t o = 0, na = 0;
        for (uint32_t e = 0; e < a.n_experts; e++) {
            a.eoff[e] = o;
            if (cnt[e]) a.active[na++] = e;
            o += cnt[e];
        }
        a.eoff[a.n_experts] = o;
        a.active[P] = na;
        nact = na;
    }
    __syncthreads();
    for (uint32_t q = threadIdx.x; q < P; q += blockDim.x) {
        const int32_t e = a.ids[q];
        if (e < 0 || (uint32_t)e >= a.n_experts) continue;
        uint32_t before = 0;
        for (uint32_t q2 = 0; q2 < q; q2++) before += a.ids[q2] == e;
        a.elist[a.eoff[e] + before] = ((q / a.topk) << 8) | (q % a.topk);
    }
    (void)nact;
}

// One round of one expert row for one lane: eight bf16 pairs (escapes patched).
template <bool R4>
__device__ __forceinline__ void moe_round(const MoeArgs &a, uint4 sv, uint2 nv, uint4 hv, uint32_t c, uint32_t b,
                                          bool act, uint8_t *escb, const uint8_t *table_s, uint32_t p[8]) {
    if (R4) {
        r4_dec16(nv, sv, a.L, p);
        if (c) {
            const uint32_t lane = lane_id();
            const uint32_t cc = c > DGT_SEG ? DGT_SEG : c;
            for (uint32_t i = lane; i < cc; i += 32) escb[i] = (uint64_t)b + i < a.n_esc ? a.esc[b + i] : 0;
            __syncwarp();
            const uint32_t m0 = act ? nib15_mask(nv.x) : 0u, m1 = act ? nib15_mask(nv.y) : 0u;
            if (!patch_escapes(p, m0, m1, cc, escb, table_s) && lane == 0) set_status(a.status, DGT_ERR_CORRUPT);
            __syncwarp();
        }
    } else {
        p[0] = sv.x; p[1] = sv.y; p[2] = sv.z; p[3] = sv.w;
        p[4] = hv.x; p[5] = hv.y; p[6] = hv.z; p[7] = hv.w;
    }
}

// A warp takes MOE_RG consecutive rows of one expert in use; for each row it
// issues the loads of up to 8 rounds at once, then walks the rounds slice by
// slice, running one fmaf chain per routed token; at the end of each slice
// the chains are butterfly-reduced and stored as that slice's partials.
constexpr uint32_t MOE_RG = 2;
constexpr uint32_t MOE_RB = 4;   // rounds loaded at once

template <bool R4>
__global__ void __launch_bounds__(MW * 32, 2) k_moe(MoeArgs a) {
    extern __shared__ uint4 xs[];  // [token][round][half][lane]
    __shared__ uint8_t table_s[256];
    __shared__ uint8_t escb[MW][DGT_SEG];
    const uint32_t tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const uint32_t K = (uint32_t)a.cols, J = a.J;
    for (uint32_t i = tid; i < a.tokens * J * 64; i += MW * 32) {
        const uint32_t t = i / (J * 64), r = i - t * J * 64;
        const uint32_t k = 8 * r, j = k >> 9, u = (k >> 4) & 31, h = (k >> 3) & 1;
        xs[(((size_t)t * J + j) * 2 + h) * 32 + u] =
            k < K ? *reinterpret_cast<const uint4 *>(a.x + (size_t)t * K + k) : make_uint4(0, 0, 0, 0);
    }
    if (R4) table_s[tid] = a.table[tid];
    __syncthreads();
    const uint32_t P = a.tokens * a.topk;
    const uint32_t nact = a.active[P];
    const uint32_t S = a.S, log2S = __ffs(S) - 1;
    const uint64_t groups = (a.ne + MOE_RG - 1) / MOE_RG;
    const uint64_t units = (uint64_t)nact * groups;
    const uint32_t Jm1 = J - 1;
    const bool last_ok = 16 * lane < K - 512 * Jm1;
    for (uint64_t uu = (uint64_t)blockIdx.x * MW + w; uu < units; uu += (uint64_t)gridDim.x * MW) {
        const uint32_t ai = (uint32_t)(uu / groups);
        const uint64_t g = uu - (uint64_t)ai * groups;
        const uint32_t e = a.active[ai];
        const uint32_t l0 = a.eoff[e], nt = a.eoff[e + 1] - l0;
        for (uint32_t tg = 0; tg < nt; tg += MOE_TPASS) {
            const uint32_t ntg = min(MOE_TPASS, nt - tg);
            const uint32_t ent = lane < ntg ? a.elist[l0 + tg + lane] : 0u;
            uint32_t tk[MOE_TPASS];
#pragma unroll
            for (int i = 0; i < (int)MOE_TPASS; i++) tk[i] = (__shfl_sync(DGT_FULL, ent, i) >> 8) % a.tokens;
            for (uint64_t r = g * MOE_RG; r < a.ne && r < (g + 1) * MOE_RG; r++) {
                const uint64_t grow = (uint64_t)e * a.ne + r;
                float acc[MOE_TPASS];
#pragma unroll
                for (int i = 0; i < (int)MOE_TPASS; i++) acc[i] = 0.0f;
                uint32_t s = 0, send = J >> log2S;  // current slice and its end round
                for (uint32_t jb = 0; jb < J; jb += MOE_RB) {
                    uint4 sv[MOE_RB], hv[MOE_RB];
                    uint2 nv[MOE_RB];
                    uint32_t sgb = 0, sgc = 0;
                    if (R4 && lane <= MOE_RB && jb + lane <= J) {
                        const uint32_t *sp = a.seg + grow * a.nseg + jb + lane;
                        sgb = sp[0];
                        sgc = jb + lane < J ? sp[1] - sgb : 0u;
                    }
#pragma unroll
                    for (uint32_t t = 0; t < MOE_RB; t++) {
                        const uint32_t j = jb + t;
                        const bool act = j < J && (j != Jm1 || last_ok);
                        const uint64_t f = grow * a.cols + (uint64_t)j * 512 + 16 * lane;
                        sv[t] = hv[t] = make_uint4(0, 0, 0, 0);
                        nv[t] = make_uint2(0, 0);
                        if (act) {
                            if (R4) {
                                sv[t] = ldg_stream16(a.sm + f);
                                nv[t] = ldg_stream8(a.nib + f / 2);
                            } else {
                                sv[t] = ldg_stream16(a.W + f);
                                hv[t] = ldg_stream16(a.W + f + 8);
                            }
                        }
                    }
#pragma unroll
                    for (uint32_t t = 0; t < MOE_RB; t++) {
                        const uint32_t j = jb + t;
                        if (j >= J) break;
                        const bool act = j != Jm1 || last_ok;
                        const uint32_t c = R4 ? __shfl_sync(DGT_FULL, sgc, t) : 0u;
                        const uint32_t b = R4 ? __shfl_sync(DGT_FULL, sgb, t) : 0u;
                        uint32_t p[8];
                        moe_round<R4>(a, sv[t], nv[t], hv[t], c, b, act, escb[w], table_s, p);
                        if (act) {
#pragma unroll
                            for (int i = 0; i < (int)MOE_TPASS; i++)
                                if ((uint32_t)i < ntg) acc[i] = fma_chunk16(p, xs + (size_t)tk[i] * J * 64, j, lane, acc[i]);
                        }
                        if (j + 1 == send) {
                            // end of slice s: reduce and store, start the next slice from +0
#pragma unroll
                            for (int i = 0; i < (int)MOE_TPASS; i++) {
                                if ((uint32_t)i < ntg) {
                                    float v = acc[i];
#pragma unroll
                                    for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(DGT_FULL, v, d);
                                    const uint32_t en = __shfl_sync(DGT_FULL, ent, i);
                                    const uint64_t q = (uint64_t)(en >> 8) * a.topk + (en & 0xFF);
                                    if (lane == 0) a.partial[(q * a.ne + r) * S + s] = v;
                                    acc[i] = 0.0f;
                                }
                            }
                            s++;
                            send = ((s + 1) * J) >> log2S;
                        }
                    }
                }
            }
        }
    }
}

__global__ void __launch_bounds__(256) k_moe_combine(MoeArgs a) {
    const uint64_t n_out = (uint64_t)a.tokens * a.ne;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_out;
         i += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t t = (uint32_t)(i / a.ne);
        const uint64_t n = i - (uint64_t)t * a.ne;
        float acc = 0.0f;
        for (uint32_t j = 0; j < a.topk; j++) {
            const uint64_t q = (uint64_t)t * a.topk + j;
            const float *pp = a.partial + (q * a.ne + n) * a.S;
            float y = pp[0];
            for (uint32_t s = 1; s < a.S; s++) y = y + pp[s];
            if (a.y32) a.y32[q * a.ne + n] = y;
            if (a.p) acc = fmaf(a.p[q], y, acc);
        }
        if (a.p) {
            if (a.out32) a.out32[i] = acc;
            if (a.out) a.out[i] = f32_to_bf16_rne(acc);
        }
    }
}

template <bool R4>
int launch_moe(MoeArgs &a, void *d_ws, size_t ws_bytes, cudaStream_t st) {
    const WsLayout l = moe_ws_layout(a.n_experts, a.ne, a.cols, a.tokens, a.topk);
    if (!d_ws || ws_bytes < l.total || ((uintptr_t)d_ws & 255)) return DGT_ERR_ARG;
    uint8_t *ws = static_cast<uint8_t *>(d_ws);
    a.eoff = reinterpret_cast<uint32_t *>(ws + l.eoff);
    a.elist = reinterpret_cast<uint32_t *>(ws + l.elist);
    a.active = reinterpret_cast<uint32_t *>(ws + l.active);
    a.partial = reinterpret_cast<float *>(ws + l.partial);
    DeviceInfo di;
    if (device_info(&di) != DGT_OK) return DGT_ERR_CUDA;
    k_moe_route<<<1, 1024, 0, st>>>(a);
    const size_t smem = (size_t)a.tokens * a.J * 1024;
    int bps = 0;
    if (prepare_kernel((const void *)k_moe<R4>, smem, MW * 32, &bps) != DGT_OK) return DGT_ERR_CUDA;
    const uint64_t pairs = (uint64_t)a.tokens * a.topk;
    const uint64_t max_units = (pairs < a.n_experts ? pairs : (uint64_t)a.n_experts) * ((a.ne + 1) / 2);
    uint64_t grid = (max_units + MW - 1) / MW;
    if (grid > (uint64_t)di.sms * bps) grid = (uint64_t)di.sms * bps;
    if (grid < 1) grid = 1;
    k_moe<R4><<<(unsigned)grid, MW * 32, smem, st>>>(a);
    const uint64_t n_out = (uint64_t)a.tokens * a.ne;
    uint64_t cgrid = (n_out + 255) / 256;
    if (cgrid > (uint64_t)di.sms * 8) cgrid = (uint64_t)di.sms * 8;
    if (cgrid < 1) cgrid = 1;
    k_moe_combine<<<(unsigned)cgrid, 256, 0, st>>>(a);
    return cudaPeekAtLastError() == cudaSuccess ? DGT_OK : DGT_ERR_CUDA;
}

static int moe_common(MoeArgs &a, uint64_t rows, uint64_t cols, uint32_t n_experts, uint32_t tokens, uint32_t topk,
                      const int32_t *d_ids, const uint16_t *d_x, const void *w_ptr, int32_t *d_status,
                      cudaStream_t st) {
    if (n_experts == 0 || n_experts > MOE_MAX_EXPERTS || rows % n_experts) return DGT_ERR_SHAPE;
    if (topk == 0 || topk > 255 || (uint64_t)tokens * topk > MOE_MAX_PAIRS || tokens >= (1u << 24))
        return DGT_ERR_SHAPE;
    if (cols == 0 || cols % 16 || cols >= (1ull << 31)) return DGT_ERR_SHAPE;
    if (!d_ids || !d_x || !w_ptr || !aligned16(d_x) || !aligned16(w_ptr)) return DGT_ERR_ARG;
    a.cols = cols;
    a.ne = rows / n_experts;
    a.n_experts = n_experts;
    a.tokens = tokens;
    a.topk = topk;
    a.J = (uint32_t)((cols + 511) / 512);
    a.S = (uint32_t)dgt_plan_slices(a.ne, cols);
    if ((uint64_t)tokens * a.J * 1024 > MOE_XS_LIMIT) return DGT_ERR_SHAPE;
    a.ids = d_ids;
    a.x = d_x;
    a.status = d_status;
    if (d_status && cudaMemsetAsync(d_status, 0, 4, st) != cudaSuccess) return DGT_ERR_CUDA;
    return DGT_OK;
}

}  // namespace dgt

using namespace dgt;

extern "C" size_t dgt_moe_workspace_bytes(uint32_t n_experts, uint64_t expert_rows, uint64_t cols, uint32_t tokens,
                                          uint32_t topk) {
    return moe_ws_layout(n_experts, expert_rows, cols, tokens, topk).total;
}

extern "C" int dgt_moe_gemv(const dgt_r4 *W, uint32_t n_experts, const int32_t *d_ids, const float *d_p,
                            uint32_t tokens, uint32_t topk, const uint16_t *d_x, float *d_y32, uint16_t *d_out,
                            float *d_out32, void *d_ws, size_t ws_bytes, int32_t *d_status, void *stream) {
    if (!W) return DGT_ERR_ARG;
    if (tokens == 0) return DGT_OK;
    cudaStream_t st = (cudaStream_t)stream;
    MoeArgs a = {};
    int rc = moe_common(a, W->rows, W->cols, n_experts, tokens, topk, d_ids, d_x, W->sm, d_status, st);
    if (rc != DGT_OK) return rc;
    if (!W->nib || !W->seg || (W->n_esc && !W->esc) || !aligned16(W->nib)) return DGT_ERR_ARG;
    a.sm = W->sm;
    a.nib = W->nib;
    a.esc = W->esc;
    a.seg = W->seg;
    a.nseg = dgt_r4_nseg(W->cols);
    a.n_esc = W->n_esc;
    a.L = make_r4lut(W->table, W->n_table);
    for (int i = 0; i < 256; i++) a.table[i] = W->table[i];
    a.p = d_p;
    a.y32 = d_y32;
    a.out = d_out;
    a.out32 = d_out32;
    return launch_moe<true>(a, d_ws, ws_bytes, st);
}

extern "C" int dgt_moe_gemv_bf16(const uint16_t *d_W, uint64_t rows, uint64_t cols, uint32_t n_experts,
                                 const int32_t *d_ids, const float *d_p, uint32_t tokens, uint32_t topk,
                                 const uint16_t *d_x, float *d_y32, uint16_t *d_out, float *d_out32, void *d_ws,
                                 size_t ws_bytes, int32_t *d_status, void *stream) {
    if (tokens == 0) return DGT_OK;
    cudaStream_t st = (cudaStream_t)stream;
    MoeArgs a = {};
    int rc = moe_common(a, rows, cols, n_experts, tokens, topk, d_ids, d_x, d_W, d_status, st);
    if (rc != DGT_OK) return rc;
    a.W = d_W;
    a.p = d_p;
    a.y32 = d_y32;
    a.out = d_out;
    a.out32 = d_out32;
    return launch_moe<false>(a, d_ws, ws_bytes, st);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of dgt_moe_gemv.
//
// Some callers cannot allocate device memory when they call: a plugin running
// inside a host framework that owns the whole device memory pool, or a
// latency-critical decode loop where a cudaMalloc (which may synchronise the
// device) is not allowed.  This entry point keeps its workspace in a fixed
// array that lives in the library's own device image, so it never calls
// cudaMalloc, cudaFree or any allocating routine.
//
// The array is DGT_MOE_NOALLOC_SCRATCH_BYTES large and every GPU that loads
// the library holds it until the process exits.  Host code cannot use the
// array's name as a device address (it is only a host-side stand-in), so the
// first call on each device, with that device current, looks the address up
// with cudaGetSymbolAddress and caches it; make that first call before any
// stream capture.  All calls share the one array and it keeps the last call's
// contents: nothing in it needs to start at zero (the routing kernel rewrites
// every list and count, and every partial sum is written before it is read),
// but calls that overlap on the GPU -- on different streams, or on
// different host threads at once -- race on it.
// ---------------------------------------------------------------------------
static __device__ __align__(256) uint8_t g_moe_scratch[DGT_MOE_NOALLOC_SCRATCH_BYTES];

static int moe_scratch_address(void **out) {
    static void *cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DGT_ERR_CUDA;
    if (!cached[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_moe_scratch) != cudaSuccess || !p) return DGT_ERR_CUDA;
        cached[dev] = p;
    }
    *out = cached[dev];
    return DGT_OK;
}

extern "C" int dgt_moe_gemv_noalloc(const dgt_r4 *W, uint32_t n_experts, const int32_t *d_ids, const float *d_p,
                                    uint32_t tokens, uint32_t topk, const uint16_t *d_x, float *d_y32,
                                    uint16_t *d_out, float *d_out32, int32_t *d_status, void *stream) {
    if (!W || n_experts == 0) return DGT_ERR_ARG;
    if (W->rows % n_experts) return DGT_ERR_SHAPE;
    if (tokens == 0) return DGT_OK;
    const size_t need = dgt_moe_workspace_bytes(n_experts, W->rows / n_experts, W->cols, tokens, topk);
    if (need > DGT_MOE_NOALLOC_SCRATCH_BYTES) return DGT_ERR_SHAPE;
    void *ws = nullptr;
    const int rc = moe_scratch_address(&ws);
    if (rc != DGT_OK) return rc;
    return dgt_moe_gemv(W, n_experts, d_ids, d_p, tokens, topk, d_x, d_y32, d_out, d_out32, ws,
                        DGT_MOE_NOALLOC_SCRATCH_BYTES, d_status, stream);
}
