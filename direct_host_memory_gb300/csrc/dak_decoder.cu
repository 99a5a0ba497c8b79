// Decode step of a Llama-shaped transformer around the direct-access operations ("DAK:
// Direct-Access-Enabled GPU Memory Offloading with Optimal Efficiency for LLM Inference",
// section 3 and section 6.1: the decode step and its time per output token; section 5:
// SplitK_GEMM replaces every nn.Linear and SplitK_FlashAttn the attention, the rest of
// the model is unchanged).
//
// Per layer, for the B requests of the step (one new token each):
//   rmsnorm   x (fp32) -> h (bf16)                         [this file]
//   dak_gemm  Wqkv . h -> qkv (fp32)
//   rope      q, k rotated; k, v appended to the cache      [this file]
//   dak_attn  q over the cache -> a (bf16)
//   dak_gemm  Wo . a -> x += (fp32)                         [added by the next rmsnorm]
//   rmsnorm   x -> h
//   dak_gemm  Wgu . h -> act = silu(gate) * up (bf16)      [fused in the GEMM's epilogue when
//                                                            Wgu is placed gate/up interleaved;
//                                                            else gu (fp32) + swiglu here]
//   dak_gemm  Wdown . act -> x +=
// and a final rmsnorm writes the output. With B <= kFuseNormMaxBatch every rmsnorm but the
// step's first and last is folded into the GEMMs around it (GemmFuse): the O and down
// projections add their product to x themselves and write h = bf16(x * g) and per-tile sums
// of x^2; gate+up and the next layer's QKV scale their accumulators by 1 / rms. With programmatic dependent launch every kernel
// starts while its predecessors drain. Before its own griddepcontrol.wait a kernel reads
// only what no kernel of the step writes (weights, KV entries older than the new token,
// the sequence lengths and the RoPE table) and writes nothing to global memory; after
// the wait its predecessor, and so every earlier kernel, has finished. The step's first
// kernel writes the sequence lengths and the RoPE table and does not signal its
// dependents, so nothing of the step starts before those are complete. In direct-access
// mode the step's kernels also hand the host link on from one to the next (LinkHandoff):
// a kernel's host tiles or requests start streaming once the earlier kernels have issued
// all of their host loads, instead of filling their rings while the previous kernel still
// streams and then idling through the boundary.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "dak_device.cuh"

struct dak_decoder {
    dak_decoder_config cfg;
    int device;
    int B;
    int n_split;
    int qkv_rows;
    std::vector<dak_decoder_layer> layers;
    const void* final_norm;
    // activations (HBM)
    float* x;              // [B][d] residual stream
    __nv_bfloat16* h;      // [B][d] normalised hidden states
    float* qkv;            // [B][(Hq + 2 Hkv) D]
    __nv_bfloat16* q;      // [B][Hq][D]
    __nv_bfloat16* att;    // [B][Hq][D]
    float* ao;             // [B][d] attention output projection
    float* gu;             // [B][2f]
    __nv_bfloat16* act;    // [B][f]
    float* dn;             // [B][d] down projection
    int* seq_lens;         // [B]
    float2* rope_cs;       // [B][D/2] (cos, sin) of the step's positions
    double* inv_freq;      // [D/2] theta^(-2i/D)
    float* ws;             // attention split workspace
    size_t ws_bytes;
    void* gemm_ws;         // the GEMMs' split workspace (this decoder's own, zeroed)
    size_t gemm_ws_bytes;
    // RMSNorms folded into the GEMMs (batch <= 128): the O and down projections add their
    // product to x and write h = bf16(x * g) and per-tile-row sums of x^2; gate+up and the
    // next QKV scale their accumulators by 1 / rms
    bool fuse_norm;
    float* ss[2];          // [T_d][B] sums of x^2 per 64 hidden units: [0] after O, [1] after down
    // host-link handoff (direct access under programmatic launch): host-tier producers of
    // the step's kernels that have issued their last load
    unsigned* link;
    // prefetch baseline
    uint8_t* staging[2];
    size_t staging_bytes;
    cudaStream_t copy_stream;
    cudaEvent_t ev_copied[2], ev_consumed[2], ev_fork, ev_join;
    // captured step
    cudaStream_t capture_stream;
    cudaGraphExec_t exec;
};

namespace dak {
namespace {

constexpr int kNormThreads = 256;
constexpr size_t kGemmWsCounterBytes = 256 * 1024;  // the counter region of a GEMM split workspace
constexpr int kNormMaxVec = 16;  // float4 per thread: d <= 16384
constexpr int kFuseNormMaxBatch = 128;  // the GEMMs' fused norm takes up to this many rows

struct NormArgs {
    float* x;                     // [B][d] residual, updated in place
    const __nv_bfloat16* x_in;    // first == 1: the step's input
    const float* delta;           // first == 0: added to x first (may be null)
    const __nv_bfloat16* g;       // gain [d]
    __nv_bfloat16* h;             // [B][d] output
    int d;
    float eps;
    // first == 1 only: per-request step set-up
    const int* positions;
    int* seq_lens;
    float2* rope_cs;
    const double* inv_freq;
    int half_d;
    int L;
    DevStatus* st;
};

// One CTA per request: x = x + delta (or the bf16 input), h = x / sqrt(mean(x^2) + eps) * g.
// The sum of squares has a fixed order (per thread, butterfly within a warp, warps in
// order), so the result does not depend on anything but the inputs.
__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const NormArgs a, const int first) {
    if (!first) grid_dep_launch();  // the first kernel lets its dependents start only when it is done
    grid_dep_wait();
    __shared__ float warp_ss[kNormThreads / 32];
    const int b = blockIdx.x;
    float* xr = a.x + static_cast<long long>(b) * a.d;
    float4 v[kNormMaxVec];
    float ss = 0.f;
    const int n4 = a.d / 4;
#pragma unroll
    for (int k = 0; k < kNormMaxVec; ++k) {
        const int j = threadIdx.x + k * kNormThreads;
        if (j < n4) {
            float4 t;
            if (first) {
                const uint2 raw = reinterpret_cast<const uint2*>(a.x_in + static_cast<long long>(b) * a.d)[j];
                const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
                const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
                t = make_float4(__low2float(lo), __high2float(lo), __low2float(hi), __high2float(hi));
            } else {
                t = reinterpret_cast<const float4*>(xr)[j];
                if (a.delta) {
                    const float4 dl = reinterpret_cast<const float4*>(a.delta + static_cast<long long>(b) * a.d)[j];
                    t.x += dl.x;
                    t.y += dl.y;
                    t.z += dl.z;
                    t.w += dl.w;
                }
            }
            if (first || a.delta) reinterpret_cast<float4*>(xr)[j] = t;
            ss += t.x * t.x + t.y * t.y + t.z * t.z + t.w * t.w;
            v[k] = t;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) warp_ss[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kNormThreads / 32; ++w) tot += warp_ss[w];
    const float r = rsqrtf(tot / static_cast<float>(a.d) + a.eps);
#pragma unroll
    for (int k = 0; k < kNormMaxVec; ++k) {
        const int j = threadIdx.x + k * kNormThreads;
        if (j < n4) {
            const uint2 graw = reinterpret_cast<const uint2*>(a.g)[j];
            const __nv_bfloat162 g01 = *reinterpret_cast<const __nv_bfloat162*>(&graw.x);
            const __nv_bfloat162 g23 = *reinterpret_cast<const __nv_bfloat162*>(&graw.y);
            const __nv_bfloat162 o01 = __floats2bfloat162_rn(v[k].x * r * __low2float(g01), v[k].y * r * __high2float(g01));
            const __nv_bfloat162 o23 = __floats2bfloat162_rn(v[k].z * r * __low2float(g23), v[k].w * r * __high2float(g23));
            uint2 out;
            out.x = *reinterpret_cast<const uint32_t*>(&o01);
            out.y = *reinterpret_cast<const uint32_t*>(&o23);
            reinterpret_cast<uint2*>(a.h + static_cast<long long>(b) * a.d)[j] = out;
        }
    }
    if (first) {
        // the step's per-request state: sequence length after the append, RoPE angles
        const int pos = a.positions[b];
        const bool ok = pos >= 0 && pos < a.L;
        if (threadIdx.x == 0) {
            a.seq_lens[b] = ok ? pos + 1 : 1;
            if (!ok) report(a.st, DAK_ERR_BOUNDS, 0xDEC0000000000000ull | static_cast<unsigned>(b));
        }
        for (int i = threadIdx.x; i < a.half_d; i += kNormThreads) {
            double s, c;
            sincos(static_cast<double>(ok ? pos : 0) * a.inv_freq[i], &s, &c);
            a.rope_cs[static_cast<long long>(b) * a.half_d + i] = make_float2(static_cast<float>(c), static_cast<float>(s));
        }
    }
}

struct RopeArgs {
    const float* qkv;          // [B][(Hq + 2 Hkv) D]
    const float2* cs;          // [B][D/2]
    const int* positions;
    __nv_bfloat16* q;          // [B][Hq][D]
    uint8_t* kv_host;          // host tier of the cache (device-visible address)
    uint8_t* kv_host_copy;     // a staged copy of the host tier to update too, or null
    uint8_t* kv_hbm;
    long long head_bytes;
    int Hq, Hkv, D, L, h_s;  // h_s: (request, kv head) slabs on the host, request-major
    DevStatus* st;
};

// grid (B, Hq + 2 Hkv), D/2 threads: thread i turns the pair (i, i + D/2) of one head.
// Query heads go to q; the new key (rotated) and value are written into the cache slab of
// their (request, kv head) at the token's row, in the cache's 16-byte-piece layout.
__global__ void __launch_bounds__(64) rope_append_kernel(const RopeArgs a) {
    grid_dep_launch();
    grid_dep_wait();
    __shared__ __align__(16) __nv_bfloat16 row[128];
    const int b = blockIdx.x, hh = blockIdx.y, i = threadIdx.x;
    const int half = a.D / 2;
    const float* src = a.qkv + (static_cast<long long>(b) * (a.Hq + 2 * a.Hkv) + hh) * a.D;
    const float x1 = src[i], x2 = src[i + half];
    float y1 = x1, y2 = x2;
    if (hh < a.Hq + a.Hkv) {
        const float2 c = a.cs[static_cast<long long>(b) * half + i];
        y1 = x1 * c.x - x2 * c.y;
        y2 = x2 * c.x + x1 * c.y;
    }
    if (hh < a.Hq) {
        __nv_bfloat16* qo = a.q + (static_cast<long long>(b) * a.Hq + hh) * a.D;
        qo[i] = __float2bfloat16_rn(y1);
        qo[i + half] = __float2bfloat16_rn(y2);
        return;
    }
    row[i] = __float2bfloat16_rn(y1);
    row[i + half] = __float2bfloat16_rn(y2);
    __syncthreads();
    const int pos = a.positions[b];
    if (pos < 0 || pos >= a.L) return;  // reported by the step's first kernel
    const bool is_v = hh >= a.Hq + a.Hkv;
    const int g = is_v ? hh - a.Hq - a.Hkv : hh - a.Hq;
    const int pieces = a.D / 8;
    if (i < pieces) {
        const uint4 piece = reinterpret_cast<const uint4*>(row)[i];
        const long long off = static_cast<long long>(pos >> 6) * (2ll * 64 * a.D * 2) + (is_v ? 64ll * a.D * 2 : 0ll) +
                              static_cast<long long>(pos & 63) * a.D * 2 + ((i ^ (pos & 7)) << 4);
        const long long slab = static_cast<long long>(b) * a.Hkv + g;
        if (slab < a.h_s) {
            const long long at = slab * a.head_bytes + off;
            *reinterpret_cast<uint4*>(a.kv_host + at) = piece;
            if (a.kv_host_copy) *reinterpret_cast<uint4*>(a.kv_host_copy + at) = piece;
        } else {
            *reinterpret_cast<uint4*>(a.kv_hbm + (slab - a.h_s) * a.head_bytes + off) = piece;
        }
    }
}

// act[b][j] = bf16(silu(gate) * up), gate = gu[b][j], up = gu[b][f + j]; f % 4 == 0.
__global__ void __launch_bounds__(256) swiglu_kernel(const float* __restrict__ gu, __nv_bfloat16* __restrict__ act,
                                                     int B, int f) {
    grid_dep_launch();
    grid_dep_wait();
    const long long n4 = static_cast<long long>(B) * f / 4;
    for (long long idx = blockIdx.x * 256ll + threadIdx.x; idx < n4; idx += static_cast<long long>(gridDim.x) * 256) {
        const long long e = idx * 4;
        const long long b = e / f;
        const long long j = e - b * f;
        const float4 g = *reinterpret_cast<const float4*>(gu + b * 2 * f + j);
        const float4 u = *reinterpret_cast<const float4*>(gu + b * 2 * f + f + j);
        const __nv_bfloat162 o01 = __floats2bfloat162_rn(g.x / (1.f + expf(-g.x)) * u.x, g.y / (1.f + expf(-g.y)) * u.y);
        const __nv_bfloat162 o23 = __floats2bfloat162_rn(g.z / (1.f + expf(-g.z)) * u.z, g.w / (1.f + expf(-g.w)) * u.w);
        uint2 out;
        out.x = *reinterpret_cast<const uint32_t*>(&o01);
        out.y = *reinterpret_cast<const uint32_t*>(&o23);
        *reinterpret_cast<uint2*>(act + e) = out;
    }
}

template <typename Kernel, typename... Args>
cudaError_t launch(Kernel k, dim3 grid, int threads, bool pdl, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, args...);
}

template <typename T>
cudaError_t dalloc(T** p, size_t count) {
    return dev_alloc(reinterpret_cast<void**>(p), std::max<size_t>(count, 1) * sizeof(T));
}

bool matrix_is(const dak_placement* p, int64_t M, int64_t K) {
    return p && p->kind == 0 && p->M == M && p->K == K && p->tile_m == kTileM;
}

// Host-resident bytes of one layer, in staging order: qkv, o, gate_up, down, kv.
const dak_placement* part(const dak_decoder_layer& L, int i) {
    switch (i) {
        case 0: return L.qkv;
        case 1: return L.o;
        case 2: return L.gate_up;
        case 3: return L.down;
        default: return L.kv;
    }
}

size_t staging_offset(const dak_decoder_layer& L, int upto) {
    size_t off = 0;
    for (int i = 0; i < upto; ++i) off += (static_cast<size_t>(part(L, i)->host_bytes) + 255) & ~size_t(255);
    return off;
}

void release(dak_decoder* d) {
    void* bufs[] = {d->x, d->h, d->qkv, d->q, d->att, d->ao, d->gu, d->act, d->dn, d->seq_lens, d->rope_cs,
                    d->inv_freq, d->ws, d->gemm_ws, d->staging[0], d->staging[1], d->ss[0], d->ss[1], d->link};
    for (void* p : bufs) dev_free(p);
    if (d->exec) cudaGraphExecDestroy(d->exec);
    for (int i = 0; i < 2; ++i) {
        if (d->ev_copied[i]) cudaEventDestroy(d->ev_copied[i]);
        if (d->ev_consumed[i]) cudaEventDestroy(d->ev_consumed[i]);
    }
    if (d->ev_fork) cudaEventDestroy(d->ev_fork);
    if (d->ev_join) cudaEventDestroy(d->ev_join);
    if (d->copy_stream) cudaStreamDestroy(d->copy_stream);
    if (d->capture_stream) cudaStreamDestroy(d->capture_stream);
}

dak_status ensure_staging(dak_decoder* d) {
    if (d->staging[0]) return DAK_OK;
    size_t need = 0;
    for (const auto& L : d->layers) need = std::max(need, staging_offset(L, 5));
    d->staging_bytes = need;
    if (need == 0) return DAK_OK;
    for (int i = 0; i < 2; ++i) {
        if (dev_alloc(reinterpret_cast<void**>(&d->staging[i]), need) != cudaSuccess) {
            cudaGetLastError();
            for (int j = 0; j < 2; ++j) {  // all or nothing: a later call tries both again
                dev_free(d->staging[j]);
                d->staging[j] = nullptr;
            }
            return DAK_ERR_DEVICE_ALLOC;
        }
    }
    return DAK_OK;
}

dak_status norm(dak_decoder* d, const NormArgs& a, int first, bool pdl, cudaStream_t s) {
    return cuda_status(launch(rmsnorm_kernel, dim3(static_cast<unsigned>(d->B)), kNormThreads, pdl, s, a, first));
}

// Copy layer l's host-resident parts into staging buffer `buf` on stream s.
dak_status prefetch_layer(dak_decoder* d, int l, uint8_t* buf, cudaStream_t s) {
    const dak_decoder_layer& L = d->layers[l];
    for (int i = 0; i < 5; ++i) {
        const dak_placement* p = part(L, i);
        if (p->host_bytes == 0) continue;
        // the device-visible alias with cudaMemcpyDefault: the form that copied fastest here
        const cudaError_t e = cudaMemcpyAsync(buf + staging_offset(L, i), p->host_dev, static_cast<size_t>(p->host_bytes),
                                              cudaMemcpyDefault, s);
        if (e != cudaSuccess) return cuda_status(e);
    }
    return DAK_OK;
}

dak_status enqueue_step(dak_decoder* d, const void* x_in, const int* positions, void* out, int mode, cudaStream_t s) {
    const dak_decoder_config& c = d->cfg;
    const bool pdl = c.plain_launch == 0;
    DevStatus* st = status_ptr();
    if (!st) return DAK_ERR_CUDA;
    dak_tuning tg[4];
    for (int i = 0; i < 4; ++i) {
        tg[i] = c.op_tuning[i];
        tg[i].pdl = pdl ? 1 : 0;
        tg[i].link = 0;  // the step runs its own handoff
    }
    dak_tuning ta = c.op_tuning[4];
    ta.n_split = d->n_split;
    ta.pdl = pdl ? 2 : 0;  // the previous kernel appends the newest token
    ta.link = 0;
    const int nl = c.n_layers;
    const int Lcap = nl > 0 ? d->layers[0].kv->L : 1;
    // the GEMMs' piece counters start every step at zero, even after a kernel that gave up
    if (d->gemm_ws &&
        cudaMemsetAsync(d->gemm_ws, 0, std::min<size_t>(d->gemm_ws_bytes, kGemmWsCounterBytes), s) != cudaSuccess)
        return DAK_ERR_CUDA;
    // Host-link handoff: each kernel's host tiles / requests start streaming once the
    // earlier kernels' host loads have all been issued (see link_wait). Every kernel of the
    // previous step has finished before the step's first one starts, so the count restarts
    // at zero here.
    const bool handoff = mode == 0 && pdl && c.no_link_handoff == 0;
    unsigned link_after = 0;
    int link_signals = 0;
    LinkHandoff lk;
    if (handoff) {
        if (cudaMemsetAsync(d->link, 0, sizeof(unsigned), s) != cudaSuccess) return DAK_ERR_CUDA;
        lk.ctr = d->link;
        lk.signals = &link_signals;
    }
    // the handoff of the next host-streaming launch, after the previous one's signals
    auto next_link = [&]() -> const LinkHandoff* {
        if (!handoff) return nullptr;
        link_after += static_cast<unsigned>(link_signals);
        link_signals = 0;
        lk.after = link_after;
        return &lk;
    };

    NormArgs na{};
    na.x = d->x;
    na.x_in = static_cast<const __nv_bfloat16*>(x_in);
    na.g = static_cast<const __nv_bfloat16*>(nl > 0 ? d->layers[0].attn_norm : d->final_norm);
    na.h = nl > 0 ? d->h : static_cast<__nv_bfloat16*>(out);
    na.d = c.hidden;
    na.eps = c.rms_eps;
    na.positions = positions;
    na.seq_lens = d->seq_lens;
    na.rope_cs = d->rope_cs;
    na.inv_freq = d->inv_freq;
    na.half_d = c.head_dim / 2;
    na.L = Lcap;
    na.st = st;
    // the step's first kernel waits for everything before it on the stream
    dak_status r = norm(d, na, 1, false, s);
    if (r != DAK_OK) return r;

    if (mode == 2) {
        if (cudaEventRecord(d->ev_fork, s) != cudaSuccess || cudaStreamWaitEvent(d->copy_stream, d->ev_fork, 0) != cudaSuccess)
            return DAK_ERR_CUDA;
        if (nl > 0) {
            if ((r = prefetch_layer(d, 0, d->staging[0], d->copy_stream)) != DAK_OK) return r;
            if (cudaEventRecord(d->ev_copied[0], d->copy_stream) != cudaSuccess) return DAK_ERR_CUDA;
        }
    }
    for (int l = 0; l < nl; ++l) {
        const dak_decoder_layer& L = d->layers[l];
        uint8_t* stg = nullptr;
        if (mode == 1) {
            stg = d->staging[0];
            if ((r = prefetch_layer(d, l, stg, s)) != DAK_OK) return r;
        } else if (mode == 2) {
            stg = d->staging[l & 1];
            if (l + 1 < nl) {
                uint8_t* nxt = d->staging[(l + 1) & 1];
                if (l >= 1 && cudaStreamWaitEvent(d->copy_stream, d->ev_consumed[(l + 1) & 1], 0) != cudaSuccess)
                    return DAK_ERR_CUDA;
                if ((r = prefetch_layer(d, l + 1, nxt, d->copy_stream)) != DAK_OK) return r;
                if (cudaEventRecord(d->ev_copied[(l + 1) & 1], d->copy_stream) != cudaSuccess) return DAK_ERR_CUDA;
            }
            if (cudaStreamWaitEvent(s, d->ev_copied[l & 1], 0) != cudaSuccess) return DAK_ERR_CUDA;
        }
        auto src = [&](int i) -> const void* {
            const dak_placement* p = part(L, i);
            if (p->host_bytes == 0) return p->host_dev;
            return stg ? static_cast<const void*>(stg + staging_offset(L, i)) : p->host_dev;
        };
        const int Hq = c.n_heads, Hkv = c.n_kv_heads, D = c.head_dim, B = d->B;
        // fused norm: the sums of squares the producing projection left, and its tile rows
        auto consumer = [&](int i) {
            GemmFuse fz;
            fz.ss_in = d->ss[i];
            fz.ss_tiles = (c.hidden + kTileM - 1) / kTileM;
            fz.inv_d = 1.f / static_cast<float>(c.hidden);
            fz.eps = c.rms_eps;
            return fz;
        };
        auto producer = [&](int i, const void* g) {
            GemmFuse fz;
            fz.res_x = d->x;
            fz.res_g = g;
            fz.ss_out = d->ss[i];
            return fz;
        };
        const GemmFuse fz_qkv = consumer(1);
        if ((r = launch_gemm(L.qkv, src(0), d->h, d->qkv, B, 1, &tg[0], s, d->gemm_ws, d->gemm_ws_bytes,
                             d->fuse_norm && l > 0 ? &fz_qkv : nullptr, next_link())) != DAK_OK)
            return r;
        RopeArgs ra{};
        ra.qkv = d->qkv;
        ra.cs = d->rope_cs;
        ra.positions = positions;
        ra.q = d->q;
        ra.kv_host = static_cast<uint8_t*>(L.kv->host_dev);
        ra.kv_host_copy = (stg && L.kv->host_bytes) ? stg + staging_offset(L, 4) : nullptr;
        ra.kv_hbm = static_cast<uint8_t*>(L.kv->hbm_ptr);
        ra.head_bytes = L.kv->head_bytes;
        ra.Hq = Hq;
        ra.Hkv = Hkv;
        ra.D = D;
        ra.L = L.kv->L;
        ra.h_s = L.kv->h_s;
        ra.st = st;
        if ((r = cuda_status(launch(rope_append_kernel, dim3(static_cast<unsigned>(B), static_cast<unsigned>(Hq + 2 * Hkv)),
                                    D / 2, pdl, s, ra))) != DAK_OK)
            return r;
        if ((r = launch_attn(d->q, L.kv, src(4), d->seq_lens, Hq, 0.f, d->att, d->ws, d->ws_bytes, &ta, s, 0,
                             next_link())) != DAK_OK)
            return r;
        if (d->fuse_norm) {
            // x += attention projection, h = bf16(x * g_mlp), sums of x^2 for gate+up
            const GemmFuse fz = producer(0, L.mlp_norm);
            if ((r = launch_gemm(L.o, src(1), d->att, d->h, B, 0, &tg[1], s, d->gemm_ws, d->gemm_ws_bytes, &fz,
                                 next_link())) != DAK_OK)
                return r;
        } else {
            if ((r = launch_gemm(L.o, src(1), d->att, d->ao, B, 1, &tg[1], s, d->gemm_ws, d->gemm_ws_bytes, nullptr,
                                 next_link())) != DAK_OK)
                return r;
            NormArgs nb{};
            nb.x = d->x;
            nb.delta = d->ao;
            nb.g = static_cast<const __nv_bfloat16*>(L.mlp_norm);
            nb.h = d->h;
            nb.d = c.hidden;
            nb.eps = c.rms_eps;
            if ((r = norm(d, nb, 0, pdl, s)) != DAK_OK) return r;
        }
        const GemmFuse fz_gu = consumer(0);
        const GemmFuse* fgu = d->fuse_norm ? &fz_gu : nullptr;
        if (L.gate_up->glu) {
            // gate/up interleaved placement: the GEMM's epilogue writes silu(gate) * up itself
            if ((r = launch_gemm(L.gate_up, src(2), d->h, d->act, B, 0, &tg[2], s, d->gemm_ws, d->gemm_ws_bytes,
                                 fgu, next_link())) != DAK_OK)
                return r;
        } else {
            if ((r = launch_gemm(L.gate_up, src(2), d->h, d->gu, B, 1, &tg[2], s, d->gemm_ws, d->gemm_ws_bytes,
                                 fgu, next_link())) != DAK_OK)
                return r;
            const long long n4 = static_cast<long long>(B) * c.ffn / 4;
            const int sg = static_cast<int>(std::min<long long>((n4 + 255) / 256, 4ll * device_sm_count()));
            if ((r = cuda_status(launch(swiglu_kernel, dim3(static_cast<unsigned>(std::max(sg, 1))), 256, pdl, s,
                                        static_cast<const float*>(d->gu), d->act, B, c.ffn))) != DAK_OK)
                return r;
        }
        const bool last = l + 1 == nl;
        if (d->fuse_norm && !last) {
            // x += down projection, h = bf16(x * g_attn of the next layer), sums for its QKV
            const GemmFuse fz = producer(1, d->layers[l + 1].attn_norm);
            if ((r = launch_gemm(L.down, src(3), d->act, d->h, B, 0, &tg[3], s, d->gemm_ws, d->gemm_ws_bytes, &fz,
                                 next_link())) != DAK_OK)
                return r;
            if (mode == 2 && cudaEventRecord(d->ev_consumed[l & 1], s) != cudaSuccess) return DAK_ERR_CUDA;
            continue;
        }
        if ((r = launch_gemm(L.down, src(3), d->act, d->dn, B, 1, &tg[3], s, d->gemm_ws, d->gemm_ws_bytes, nullptr,
                             next_link())) != DAK_OK)
            return r;
        if (mode == 2 && cudaEventRecord(d->ev_consumed[l & 1], s) != cudaSuccess) return DAK_ERR_CUDA;
        NormArgs nc{};
        nc.x = d->x;
        nc.delta = d->dn;
        nc.g = static_cast<const __nv_bfloat16*>(last ? d->final_norm : d->layers[l + 1].attn_norm);
        nc.h = last ? static_cast<__nv_bfloat16*>(out) : d->h;
        nc.d = c.hidden;
        nc.eps = c.rms_eps;
        if ((r = norm(d, nc, 0, pdl && mode != 2, s)) != DAK_OK) return r;
    }
    if (mode == 2) {
        if (cudaEventRecord(d->ev_join, d->copy_stream) != cudaSuccess || cudaStreamWaitEvent(s, d->ev_join, 0) != cudaSuccess)
            return DAK_ERR_CUDA;
    }
    return DAK_OK;
}

}  // namespace
}  // namespace dak

using namespace dak;

extern "C" dak_status dak_decoder_create(const dak_decoder_config* cfg, const dak_decoder_layer* layers,
                                         const void* final_norm, dak_decoder** out) {
    if (!out) return DAK_ERR_INVALID;
    *out = nullptr;
    if (!cfg || !final_norm || cfg->n_layers < 0 || (cfg->n_layers > 0 && !layers)) return DAK_ERR_INVALID;
    dak_decoder_config c = *cfg;
    if (c.rms_eps <= 0.f) c.rms_eps = 1e-5f;
    if (c.rope_theta <= 0.f) c.rope_theta = 500000.f;
    if (c.hidden <= 0 || c.n_heads <= 0 || c.n_kv_heads <= 0 || c.ffn <= 0 || c.n_heads % c.n_kv_heads)
        return DAK_ERR_INVALID;
    if (c.head_dim != 64 && c.head_dim != 128) return DAK_ERR_UNSUPPORTED;
    if (c.hidden % 8 || c.ffn % 8) return DAK_ERR_ALIGN;
    if (c.hidden > 4 * kNormThreads * kNormMaxVec) return DAK_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(final_norm) & 15)) return DAK_ERR_ALIGN;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DAK_ERR_CUDA;
    const int64_t d = c.hidden, D = c.head_dim, f = c.ffn;
    const int64_t qkv_rows = (c.n_heads + 2 * static_cast<int64_t>(c.n_kv_heads)) * D;
    int B = 0, Lcap = 0;
    for (int l = 0; l < c.n_layers; ++l) {
        const dak_decoder_layer& L = layers[l];
        if (!matrix_is(L.qkv, qkv_rows, d) || !matrix_is(L.o, d, c.n_heads * D) || !matrix_is(L.gate_up, 2 * f, d) ||
            !matrix_is(L.down, d, f))
            return DAK_ERR_INVALID;
        if (!L.kv || L.kv->kind != 1 || L.kv->H_kv != c.n_kv_heads || L.kv->D != c.head_dim) return DAK_ERR_INVALID;
        if (!L.attn_norm || !L.mlp_norm) return DAK_ERR_INVALID;
        if ((reinterpret_cast<uintptr_t>(L.attn_norm) & 15) || (reinterpret_cast<uintptr_t>(L.mlp_norm) & 15))
            return DAK_ERR_ALIGN;
        if (l == 0) {
            B = L.kv->B;
            Lcap = L.kv->L;
        }
        if (L.kv->B != B || L.kv->L != Lcap) return DAK_ERR_INVALID;
        const dak_placement* parts[] = {L.qkv, L.o, L.gate_up, L.down, L.kv};
        for (const dak_placement* p : parts)
            if (p->device != dev) return DAK_ERR_INVALID;
    }
    if (c.n_layers == 0) B = 1;

    dak_decoder* dd = new dak_decoder();
    dd->cfg = c;
    dd->device = dev;
    dd->B = B;
    dd->qkv_rows = static_cast<int>(qkv_rows);
    dd->layers.assign(layers, layers + c.n_layers);
    dd->final_norm = final_norm;
    dd->n_split = c.op_tuning[4].n_split > 0 ? c.op_tuning[4].n_split
                                              : (c.n_layers > 0 ? dak_attn_default_split(layers[0].kv) : 1);
    const size_t Bs = static_cast<size_t>(B);
    cudaError_t e = cudaSuccess;
    auto chk = [&](cudaError_t x) {
        if (e == cudaSuccess) e = x;
    };
    chk(dalloc(&dd->x, Bs * d));
    chk(dalloc(&dd->h, Bs * d));
    chk(dalloc(&dd->qkv, Bs * qkv_rows));
    chk(dalloc(&dd->q, Bs * c.n_heads * D));
    chk(dalloc(&dd->att, Bs * c.n_heads * D));
    chk(dalloc(&dd->ao, Bs * d));
    chk(dalloc(&dd->gu, Bs * 2 * f));
    chk(dalloc(&dd->act, Bs * f));
    chk(dalloc(&dd->dn, Bs * d));
    chk(dalloc(&dd->seq_lens, Bs));
    chk(dalloc(&dd->rope_cs, Bs * D / 2));
    chk(dalloc(&dd->inv_freq, static_cast<size_t>(D / 2)));
    chk(dalloc(&dd->link, 1));
    dd->ws_bytes = dak_attn_workspace_bytes(B, c.n_heads, c.head_dim, dd->n_split);
    if (dd->ws_bytes) chk(dev_alloc(reinterpret_cast<void**>(&dd->ws), dd->ws_bytes));
    // a split workspace of its own, so that decoders on different streams never share one
    dd->gemm_ws_bytes = 0;
    for (int l = 0; l < c.n_layers; ++l)
        for (const dak_placement* g : {layers[l].qkv, layers[l].o, layers[l].gate_up, layers[l].down})
            dd->gemm_ws_bytes = std::max(dd->gemm_ws_bytes, gemm_workspace_bytes(g, B));
    if (dd->gemm_ws_bytes) {
        chk(dev_alloc(&dd->gemm_ws, dd->gemm_ws_bytes));
        if (e == cudaSuccess) chk(cudaMemset(dd->gemm_ws, 0, dd->gemm_ws_bytes));
    }
    dd->fuse_norm = B <= kFuseNormMaxBatch;
    if (dd->fuse_norm) {
        const size_t ss_bytes = static_cast<size_t>((d + kTileM - 1) / kTileM) * B * sizeof(float);
        for (int i = 0; i < 2; ++i) chk(dev_alloc(reinterpret_cast<void**>(&dd->ss[i]), ss_bytes));
    }
    if (e == cudaSuccess) {
        std::vector<double> inv(D / 2);
        for (int64_t i = 0; i < D / 2; ++i)
            inv[i] = std::pow(static_cast<double>(c.rope_theta), -2.0 * static_cast<double>(i) / static_cast<double>(D));
        chk(cudaMemcpy(dd->inv_freq, inv.data(), inv.size() * sizeof(double), cudaMemcpyHostToDevice));
    }
    chk(cudaStreamCreateWithFlags(&dd->copy_stream, cudaStreamNonBlocking));
    chk(cudaStreamCreateWithFlags(&dd->capture_stream, cudaStreamNonBlocking));
    for (int i = 0; i < 2; ++i) {
        chk(cudaEventCreateWithFlags(&dd->ev_copied[i], cudaEventDisableTiming));
        chk(cudaEventCreateWithFlags(&dd->ev_consumed[i], cudaEventDisableTiming));
    }
    chk(cudaEventCreateWithFlags(&dd->ev_fork, cudaEventDisableTiming));
    chk(cudaEventCreateWithFlags(&dd->ev_join, cudaEventDisableTiming));
    if (e != cudaSuccess) {
        cudaGetLastError();
        release(dd);
        delete dd;
        return e == cudaErrorMemoryAllocation ? DAK_ERR_DEVICE_ALLOC : DAK_ERR_CUDA;
    }
    *out = dd;
    return DAK_OK;
}

extern "C" int dak_decoder_batch(const dak_decoder* dec) { return dec ? dec->B : 0; }

extern "C" dak_status dak_decoder_step(dak_decoder* dec, const void* x_in, const int* positions, void* out, int mode,
                                       void* stream) {
    if (!dec || !x_in || !positions || !out || mode < 0 || mode > 2) return DAK_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(x_in) & 15) || (reinterpret_cast<uintptr_t>(out) & 15)) return DAK_ERR_ALIGN;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DAK_ERR_CUDA;
    if (dev != dec->device) return DAK_ERR_INVALID;
    if (mode != 0) {
        const dak_status r = ensure_staging(dec);
        if (r != DAK_OK) return r;
    }
    return enqueue_step(dec, x_in, positions, out, mode, static_cast<cudaStream_t>(stream));
}

extern "C" dak_status dak_decoder_capture(dak_decoder* dec, const void* x_in, const int* positions, void* out,
                                          int mode) {
    if (!dec || !x_in || !positions || !out || mode < 0 || mode > 2) return DAK_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(x_in) & 15) || (reinterpret_cast<uintptr_t>(out) & 15)) return DAK_ERR_ALIGN;
    if (mode != 0) {
        const dak_status r = ensure_staging(dec);
        if (r != DAK_OK) return r;
    }
    if (!status_ptr()) return DAK_ERR_CUDA;  // look the status block up outside the capture
    if (dec->exec) {
        cudaGraphExecDestroy(dec->exec);
        dec->exec = nullptr;
    }
    cudaStream_t s = dec->capture_stream;
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
        cudaGetLastError();
        return DAK_ERR_CUDA;
    }
    const dak_status r = enqueue_step(dec, x_in, positions, out, mode, s);
    cudaGraph_t g = nullptr;
    const cudaError_t e = cudaStreamEndCapture(s, &g);
    if (r != DAK_OK || e != cudaSuccess) {
        cudaGetLastError();
        if (g) cudaGraphDestroy(g);
        return r != DAK_OK ? r : DAK_ERR_CUDA;
    }
    const cudaError_t ei = cudaGraphInstantiate(&dec->exec, g, 0);
    cudaGraphDestroy(g);
    if (ei != cudaSuccess) {
        cudaGetLastError();
        dec->exec = nullptr;
        return DAK_ERR_CUDA;
    }
    return DAK_OK;
}

extern "C" dak_status dak_decoder_replay(dak_decoder* dec, void* stream) {
    if (!dec || !dec->exec) return DAK_ERR_INVALID;
    return cuda_status(cudaGraphLaunch(dec->exec, static_cast<cudaStream_t>(stream)));
}

extern "C" int dak_decoder_launches(const dak_decoder* dec, int mode) {
    (void)mode;
    if (!dec) return 0;
    int n = 1;
    // per layer: QKV, RoPE + append, attention (+ split merge), O, gate+up (+ SwiGLU), down and
    // two RMSNorms, of which a fused decoder keeps only the step's last
    for (const auto& L : dec->layers) n += 6 + (dec->n_split > 1 ? 1 : 0) + (L.gate_up->glu ? 0 : 1) + (dec->fuse_norm ? 0 : 2);
    if (dec->fuse_norm && !dec->layers.empty()) n += 1;
    return n;
}

extern "C" dak_status dak_decoder_free(dak_decoder* dec) {
    if (!dec) return DAK_OK;
    cudaDeviceSynchronize();
    release(dec);
    delete dec;
    return DAK_OK;
}
