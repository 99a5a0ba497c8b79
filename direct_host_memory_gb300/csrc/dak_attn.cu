// SplitK_FlashAttn for decode: single-query GQA attention over a KV cache whose requests
// are split between pinned, device-mapped host memory and HBM ("DAK: Direct-Access-Enabled
// GPU Memory Offloading with Optimal Efficiency for LLM Inference", section 5, "Supporting
// FlashAttention"). Each request attends wholly within one tier.
//
// Work unit = (request, kv head, context split). The split count is fixed per call and
// does not depend on the placement, so results are identical for every offload ratio.
// Persistent CTAs [0, n_host) take the host units, the rest the HBM units; inside a CTA a
// producer thread streams 64-token chunks of K and V into a shared-memory ring with bulk
// asynchronous copies, and four consumer warps each own 16 tokens of every chunk.
//
// The contractions are tiny (the M side is the G = Hq/Hkv query heads sharing a kv head),
// so they run on warp-level m16n8k16 MMAs rather than the tcgen05 pipeline:
//   S  = Q_g (16 x D, rows >= G zero) . K^T (D x 16 tokens)
//   O += P   (16 x 16 tokens)         . V   (16 tokens x D)
// with online softmax in fp32 (base-2 exponentials, the scale folded with log2 e). The
// MMA takes bf16 operands, so the fp32 probabilities P enter the second product as bf16.
// With a bf16 output (dak_attn) that is one bf16(P): its rounding (2^-9 relative per
// probability, averaging out over the tokens) stays below the output's own rounding. With
// an fp32 output (dak_attn_f32, the parity mode) P enters as two bf16 parts, P_hi = bf16(P)
// and P_lo = bf16(P - P_hi), multiplied into the same fp32 accumulators: P_hi + P_lo equals
// P to about 2^-17 relative (the second set of P.V MMAs costs 4% on an all-HBM launch with
// 8 query heads per kv head). The denominator always sums the fp32 P.
// Partial results of the splits are merged by a log-sum-exp combine in fixed order.
//
// KV placement layout: per tier [requests][H_kv] slabs; a slab is ceil(L/64) chunks of 64
// tokens stored [K 64 x D][V 64 x D] bf16 (last chunk zero-padded), so that one bulk copy
// brings a whole stage; inside every token row the 16-byte piece c sits at c ^ (token & 7)
// so that ldmatrix reads of 8 consecutive tokens hit 8 different bank groups.
#include <algorithm>
#include <cmath>

#include "dak_device.cuh"

namespace dak {

struct AttnParams {
    const __nv_bfloat16* Q;  // [B][Hq][D]
    const uint8_t* kv[2];    // [0] host tier (device-visible), [1] HBM tier
    const int* seq_lens;
    void* O;                 // [B][Hq][D], bf16 or (o_fp32) fp32
    int o_fp32;
    float* ws;               // [B][Hq][n_split][D + 2] partials: m (log2 domain), l, o[D]
    int B, Hq, Hkv, G, L, h_s, n_split, split_len;  // h_s: host slabs (request-major)
    int wait_newest;         // stream the chunk holding token L_b - 1 only after the previous kernel
    float scale_log2;
    long long head_bytes;    // bytes of one (request, kv head) slab
    int n_host_ctas, n_hbm_ctas, host_window, hbm_window;
    long long host_units, hbm_units;
    DevStatus* st;
    // host-link handoff of a decode step (link_wait / link_signal; null = off)
    unsigned* link;
    unsigned link_after;
};

constexpr int kChunkTok = 64;
constexpr int kAttnConsumers = 4;
constexpr int kAttnThreads = 32 * (1 + kAttnConsumers);

struct UnitRange {
    int tier;
    long long begin, end;  // global unit indices
    int window;
};

__device__ __forceinline__ UnitRange units_of_cta(const AttnParams& p) {
    UnitRange u;
    const int b = blockIdx.x;
    if (b < p.n_host_ctas) {
        u.tier = 0;
        u.begin = p.host_units * b / p.n_host_ctas;
        u.end = p.host_units * (b + 1) / p.n_host_ctas;
        u.window = p.host_window;
    } else {
        const int j = b - p.n_host_ctas;
        u.tier = 1;
        u.begin = p.host_units + p.hbm_units * j / p.n_hbm_ctas;
        u.end = p.host_units + p.hbm_units * (j + 1) / p.n_hbm_ctas;
        u.window = p.hbm_window;
    }
    return u;
}

struct Unit {
    int b, g, s;
    int t0, t1;  // token range
    int Lb;      // tokens of the request
    const uint8_t* base;  // the (request, kv head) slab
};

__device__ __forceinline__ Unit decode_unit(const AttnParams& p, long long u, int tier) {
    Unit x;
    const int per_b = p.Hkv * p.n_split;
    x.b = static_cast<int>(u / per_b);
    const int rem = static_cast<int>(u - static_cast<long long>(x.b) * per_b);
    x.g = rem / p.n_split;
    x.s = rem - x.g * p.n_split;
    int Lb = p.L;
    if (p.seq_lens) Lb = min(max(p.seq_lens[x.b], 0), p.L);
    x.Lb = Lb;
    x.t0 = x.s * p.split_len;
    x.t1 = min(Lb, x.t0 + p.split_len);
    const long long slab = static_cast<long long>(x.b) * p.Hkv + x.g;  // its index in the tier
    x.base = p.kv[tier] + (tier == 0 ? slab : slab - p.h_s) * p.head_bytes;
    return x;
}

enum : uint32_t { A_PROD_EMPTY = 11, A_CONS_FULL = 12, A_DRAIN = 13 };

// One output element, bf16 (round to nearest even) or fp32.
__device__ __forceinline__ void store_out(void* O, int o_fp32, long long i, float v) {
    if (o_fp32) {
        static_cast<float*>(O)[i] = v;
    } else {
        static_cast<__nv_bfloat16*>(O)[i] = __float2bfloat16_rn(v);
    }
}

// Two fp32 values as the bf16 pairs hi = bf16(v) and lo = bf16(v - hi) (round to nearest even).
__device__ __forceinline__ void split_bf16(float v0, float v1, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat16 h0 = __float2bfloat16_rn(v0), h1 = __float2bfloat16_rn(v1);
    hi = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) | (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
    lo = pack_bf16(v0 - __bfloat162float(h0), v1 - __bfloat162float(h1));
}

__device__ __forceinline__ void named_bar_consumers() {
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kAttnConsumers) : "memory");
}

template <int D, bool SPLIT_P>
__global__ void __launch_bounds__(kAttnThreads, 2) attn_kernel(const AttnParams p) {
    constexpr int KS = D / 16;                       // k-steps of the score MMA
    constexpr int NB = D / 8;                        // 8-wide column blocks of O
    constexpr int CHUNK_BYTES = kChunkTok * D * 2;   // K (or V) bytes of one chunk
    constexpr int STAGE = 2 * CHUNK_BYTES;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t full[8], empty[8];
    __shared__ int abort_flag;
    volatile int* abort = &abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const UnitRange ur = units_of_cta(p);
    const int W = ur.window;
    float* comb = reinterpret_cast<float*>(smem + static_cast<size_t>(W) * STAGE);  // [4 warps][G][D + 2]

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < W; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kAttnConsumers);
        }
        fence_mbar_init();
    }
    __syncthreads();
    grid_dep_launch();

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            const bool link = ur.tier == 0 && p.link;
            if (link) link_wait(p.link, p.link_after, p.st);
            long long i = 0;
            bool waited = false;
            for (long long u = ur.begin; u < ur.end && !*abort; ++u) {
                const Unit x = decode_unit(p, u, ur.tier);
                for (int t = x.t0; t < x.t1; t += kChunkTok, ++i) {
                    const int s = static_cast<int>(i % W);
                    if (p.wait_newest && !waited && t + kChunkTok >= x.Lb) {
                        grid_dep_wait();  // this chunk holds the newest token, which the previous kernel writes
                        waited = true;
                    }
                    if (i >= W && !mbar_wait(&empty[s], static_cast<uint32_t>(((i / W) - 1) & 1), abort, p.st,
                                             DAK_ERR_TIMEOUT, A_PROD_EMPTY)) {
                        goto producer_done;
                    }
                    uint8_t* dst = smem + static_cast<size_t>(s) * STAGE;
                    mbar_arrive_expect_tx(&full[s], STAGE);
                    bulk_g2s(dst, x.base + static_cast<long long>(t / kChunkTok) * STAGE, STAGE, &full[s], pol);
                }
            }
        producer_done:
            if (link) link_signal(p.link);
            volatile int dummy = 0;
            for (int s = 0; s < W && s < i; ++s) {
                const long long last = ((i - 1 - s) / W) * W + s;
                mbar_wait(&full[s], static_cast<uint32_t>((last / W) & 1), &dummy, p.st, DAK_ERR_TIMEOUT, A_DRAIN);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // Q (and the outputs) may belong to the previous kernel of the stream; the KV cache
    // streamed above is, with programmatic launch, taken to be written earlier than that
    grid_dep_wait();
    const int w = warp - 1;
    const int q4 = lane & 3;      // column pair within an 8-wide block
    const int ra = lane >> 2;     // MMA row of c0/c1 (c2/c3: ra + 8)
    const int mi = lane >> 3, rr = lane & 7;  // ldmatrix: matrix index, row within it
    long long i = 0;
    bool failed = false;  // a wait ran out: skip the math but keep meeting the named barriers
    for (long long u = ur.begin; u < ur.end; ++u) {
        const Unit x = decode_unit(p, u, ur.tier);
        // Q fragments (A operand), rows >= G are zero
        uint32_t qa[KS][4];
        {
            const __nv_bfloat16* qb = p.Q + (static_cast<long long>(x.b) * p.Hq + static_cast<long long>(x.g) * p.G) * D;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int k = ks * 16 + 2 * q4;
                qa[ks][0] = ra < p.G ? *reinterpret_cast<const uint32_t*>(qb + ra * D + k) : 0u;
                qa[ks][1] = ra + 8 < p.G ? *reinterpret_cast<const uint32_t*>(qb + (ra + 8) * D + k) : 0u;
                qa[ks][2] = ra < p.G ? *reinterpret_cast<const uint32_t*>(qb + ra * D + k + 8) : 0u;
                qa[ks][3] = ra + 8 < p.G ? *reinterpret_cast<const uint32_t*>(qb + (ra + 8) * D + k + 8) : 0u;
            }
        }
        float o[NB][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;
        float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

        for (int t = x.t0; t < x.t1; t += kChunkTok, ++i) {
            const int s = static_cast<int>(i % W);
            if (!failed && !mbar_wait(&full[s], static_cast<uint32_t>((i / W) & 1), abort, p.st, DAK_ERR_TIMEOUT,
                                      A_CONS_FULL)) {
                failed = true;
            }
            if (failed) continue;
            const int valid = min(kChunkTok, x.t1 - t) - 16 * w;  // tokens of this warp's 16 that are real
            if (valid > 0) {
                const uint32_t ks_base = smem_u32(smem + static_cast<size_t>(s) * STAGE);
                const uint32_t vs_base = ks_base + CHUNK_BYTES;
                // ---- scores: 16 rows x 16 tokens
                float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                {
                    const int tok = 16 * w + (mi >> 1) * 8 + rr;
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        const int c = ks * 2 + (mi & 1);
                        const uint32_t addr = ks_base + static_cast<uint32_t>(tok * D * 2 + ((c ^ (tok & 7)) << 4));
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(addr, b0, b1, b2, b3);
                        mma_bf16_16816(sc[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
                        mma_bf16_16816(sc[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
                    }
                }
                // ---- scale, mask, online softmax (rows ra and ra + 8)
                float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
                for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int tk = nb * 8 + 2 * q4 + e;
                        const bool ok = tk < valid;
                        sc[nb][e] = ok ? sc[nb][e] * p.scale_log2 : -INFINITY;
                        sc[nb][2 + e] = ok ? sc[nb][2 + e] * p.scale_log2 : -INFINITY;
                        mx_a = fmaxf(mx_a, sc[nb][e]);
                        mx_b = fmaxf(mx_b, sc[nb][2 + e]);
                    }
                }
                mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
                mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
                mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
                mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
                const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
                const float base_a = mn_a == -INFINITY ? 0.f : mn_a;
                const float base_b = mn_b == -INFINITY ? 0.f : mn_b;
                const float corr_a = exp2f(m_a - base_a), corr_b = exp2f(m_b - base_b);
                m_a = mn_a;
                m_b = mn_b;
                float pr[2][4];
                float ps_a = 0.f, ps_b = 0.f;
#pragma unroll
                for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        pr[nb][e] = exp2f(sc[nb][e] - base_a);
                        pr[nb][2 + e] = exp2f(sc[nb][2 + e] - base_b);
                        ps_a += pr[nb][e];
                        ps_b += pr[nb][2 + e];
                    }
                }
                l_a = l_a * corr_a + ps_a;
                l_b = l_b * corr_b + ps_b;
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                    o[nb][0] *= corr_a;
                    o[nb][1] *= corr_a;
                    o[nb][2] *= corr_b;
                    o[nb][3] *= corr_b;
                }
                // P as the A operand (16 rows x 16 tokens): hi = bf16(P), and with SPLIT_P also
                // lo = bf16(P - hi), both multiplied into the same accumulators
                uint32_t pa0, pa1, pa2, pa3, pl0, pl1, pl2, pl3;
                split_bf16(pr[0][0], pr[0][1], pa0, pl0);
                split_bf16(pr[0][2], pr[0][3], pa1, pl1);
                split_bf16(pr[1][0], pr[1][1], pa2, pl2);
                split_bf16(pr[1][2], pr[1][3], pa3, pl3);
                // ---- O += P V
                {
                    const int tok = 16 * w + (mi & 1) * 8 + rr;
#pragma unroll
                    for (int db = 0; db < NB / 2; ++db) {
                        const int c = db * 2 + (mi >> 1);
                        const uint32_t addr = vs_base + static_cast<uint32_t>(tok * D * 2 + ((c ^ (tok & 7)) << 4));
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(addr, b0, b1, b2, b3);
                        mma_bf16_16816(o[2 * db], pa0, pa1, pa2, pa3, b0, b1);
                        mma_bf16_16816(o[2 * db + 1], pa0, pa1, pa2, pa3, b2, b3);
                        if (SPLIT_P) {
                            mma_bf16_16816(o[2 * db], pl0, pl1, pl2, pl3, b0, b1);
                            mma_bf16_16816(o[2 * db + 1], pl0, pl1, pl2, pl3, b2, b3);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }

        // ---- merge the four warps' partial states (fixed order), then write
        l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
        l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
        float* cw = comb + static_cast<size_t>(w) * p.G * (D + 2);
        if (ra < p.G) {
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                const int d = nb * 8 + 2 * q4;
                cw[ra * (D + 2) + d] = o[nb][0];
                cw[ra * (D + 2) + d + 1] = o[nb][1];
            }
            if (q4 == 0) {
                cw[ra * (D + 2) + D] = m_a;
                cw[ra * (D + 2) + D + 1] = l_a;
            }
        }
        if (ra + 8 < p.G) {
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                const int d = nb * 8 + 2 * q4;
                cw[(ra + 8) * (D + 2) + d] = o[nb][2];
                cw[(ra + 8) * (D + 2) + d + 1] = o[nb][3];
            }
            if (q4 == 0) {
                cw[(ra + 8) * (D + 2) + D] = m_b;
                cw[(ra + 8) * (D + 2) + D + 1] = l_b;
            }
        }
        named_bar_consumers();
        const int ctid = threadIdx.x - 32;
        for (int e = ctid; e < p.G * D; e += 32 * kAttnConsumers) {
            const int r = e / D, d = e - r * D;
            float M = -INFINITY;
#pragma unroll
            for (int ww = 0; ww < kAttnConsumers; ++ww) M = fmaxf(M, comb[(ww * p.G + r) * (D + 2) + D]);
            const float base = M == -INFINITY ? 0.f : M;
            float acc = 0.f, lsum = 0.f;
#pragma unroll
            for (int ww = 0; ww < kAttnConsumers; ++ww) {
                const float* row = comb + (ww * p.G + r) * (D + 2);
                const float f = exp2f(row[D] - base);
                acc += f * row[d];
                lsum += f * row[D + 1];
            }
            const long long orow = static_cast<long long>(x.b) * p.Hq + static_cast<long long>(x.g) * p.G + r;
            if (p.n_split == 1) {
                store_out(p.O, p.o_fp32, orow * D + d, lsum > 0.f ? acc / lsum : 0.f);
            } else {
                float* wr = p.ws + (orow * p.n_split + x.s) * (D + 2);
                wr[d] = acc;
                if (d == 0) {
                    wr[D] = M;
                    wr[D + 1] = lsum;
                }
            }
        }
        named_bar_consumers();  // comb is rewritten by the next unit
    }
}

// Merge the context splits of every (request, query head) row in split order:
//   o = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s,  M = max_s m_s.
// Two forms; the order of every sum depends on the split count alone.
//
// A few splits: one warp per row walks the splits in order (lanes over the columns).
template <int D>
__global__ void attn_combine_warp_kernel(const float* __restrict__ ws, void* __restrict__ O, int o_fp32, int rows,
                                         int n_split) {
    grid_dep_launch();
    grid_dep_wait();  // the partials come from the attention kernel just before
    const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float* base = ws + static_cast<long long>(row) * n_split * (D + 2);
    float M = -INFINITY;
    for (int s = 0; s < n_split; ++s) M = fmaxf(M, base[s * (D + 2) + D]);
    const float mb = M == -INFINITY ? 0.f : M;
    float lsum = 0.f;
    float acc[D / 32];
#pragma unroll
    for (int j = 0; j < D / 32; ++j) acc[j] = 0.f;
    for (int s = 0; s < n_split; ++s) {
        const float* ps = base + s * (D + 2);
        const float f = exp2f(ps[D] - mb);
        lsum += f * ps[D + 1];
#pragma unroll
        for (int j = 0; j < D / 32; ++j) acc[j] += f * ps[lane + 32 * j];
    }
#pragma unroll
    for (int j = 0; j < D / 32; ++j) {
        store_out(O, o_fp32, static_cast<long long>(row) * D + lane + 32 * j, lsum > 0.f ? acc[j] / lsum : 0.f);
    }
}

// Many splits: one CTA per row. The threads take the splits side by side (the maxima,
// then the factors and the denominator, then column pairs of o_s in groups of splits), so
// that every phase is one round trip to L2 whatever the split count; the groups' partial
// sums are added in group order. (One request over a 4K context: the attention with 16
// splits 10.7 -> 8.4 us, with 32 splits 13.7 -> 7.1 us; at 2 and 4 splits the warp form
// is 0.5 us faster.)
constexpr int kCombineThreads = 256;
constexpr int kCombineWarpMaxSplits = 4;
constexpr int kMaxSplits = 1024;

template <int D>
__global__ void __launch_bounds__(kCombineThreads) attn_combine_cta_kernel(const float* __restrict__ ws,
                                                                           void* __restrict__ O, int o_fp32,
                                                                           int n_split) {
    constexpr int CG = D / 2;                   // float2 column pairs of a row
    constexpr int SG = kCombineThreads / CG;    // groups of splits
    constexpr int NW = kCombineThreads / 32;
    __shared__ float fs[kMaxSplits];
    __shared__ float red[SG][D];
    __shared__ float wred[2][NW];
    grid_dep_launch();
    grid_dep_wait();  // the partials come from the attention kernel just before
    const int row = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float* base = ws + static_cast<long long>(row) * n_split * (D + 2);
    float M = -INFINITY;
    for (int s = tid; s < n_split; s += kCombineThreads) M = fmaxf(M, base[s * (D + 2) + D]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (lane == 0) wred[0][warp] = M;
    __syncthreads();
    M = wred[0][0];
#pragma unroll
    for (int w = 1; w < NW; ++w) M = fmaxf(M, wred[0][w]);
    const float mb = M == -INFINITY ? 0.f : M;
    float l = 0.f;
    for (int s = tid; s < n_split; s += kCombineThreads) {
        const float f = exp2f(base[s * (D + 2) + D] - mb);
        fs[s] = f;
        l += f * base[s * (D + 2) + D + 1];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) wred[1][warp] = l;
    __syncthreads();
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) lsum += wred[1][w];
    const int c = tid % CG, g = tid / CG;
    float ax = 0.f, ay = 0.f;
#pragma unroll 8
    for (int s = g; s < n_split; s += SG) {
        const float2 v = *reinterpret_cast<const float2*>(base + s * (D + 2) + 2 * c);
        ax += fs[s] * v.x;
        ay += fs[s] * v.y;
    }
    red[g][2 * c] = ax;
    red[g][2 * c + 1] = ay;
    __syncthreads();
    for (int d = tid; d < D; d += kCombineThreads) {
        float acc = 0.f;
#pragma unroll
        for (int gg = 0; gg < SG; ++gg) acc += red[gg][d];
        store_out(O, o_fp32, static_cast<long long>(row) * D + d, lsum > 0.f ? acc / lsum : 0.f);
    }
}

constexpr int kAttnDefaultHostCtas = 32;
constexpr int kAttnDefaultHostWindow = 4;
// Default ring depth: 2 stages (64 KiB in flight per CTA; three CTAs fit on an SM). Measured
// all in HBM, graphs of back-to-back launches: 32 requests x 8 kv heads over 8K context (4
// MiB units) 0.89-0.91 of B_hbm with 3 stages, 0.97 with 2 (more copies in flight only queue
// in the memory system); 16 x 8 over 4K in two splits 0.82-0.83 either way; with host
// requests the link bounds both alike.
constexpr int kAttnStages = 2;
constexpr int kAttnMaxStages = 5;

// Context splits: double the split count while the units fill less than about 80% of the
// CTA slots (two CTAs per SM) and a split keeps at least 128 tokens. With every CTA
// streaming at the same rate, more splits add no token-waves of parallelism, only partial
// results to merge (measured: 32 requests x 8 kv heads over 8K context ran 1.3% faster
// unsplit than with 4 splits; one request over 4K context ran 7.1 us with 32 splits of 128
// tokens, 8.4 with 16 of 256, 9.0 with 64).
static int default_split(int B, int Hkv, int L) {
    const long long slots = 2ll * device_sm_count();
    int n = 1;
    while (static_cast<long long>(B) * Hkv * n * 5 < slots * 4 && n * 2 * 128 <= L && n < 64) n *= 2;
    return n;
}

template <int D>
static int attn_smem_bytes(int W, int G) {
    return W * 2 * kChunkTok * D * 2 + kAttnConsumers * G * (D + 2) * 4;
}

// CTAs of this kernel that fit on one SM with the given ring depth (each CTA streams its own
// copies, so two per SM double the copy streams an SM keeps in flight).
template <int D>
static int attn_ctas_per_sm(int W, int G) {
    int n = 0;
    const int smem = attn_smem_bytes<D>(W, G);
    if (cudaFuncSetAttribute(attn_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_kernel<D, false>, kAttnThreads, smem) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    return std::max(1, n);
}

// Launch with or without programmatic dependent launch (the kernel may start while the
// previous kernel of the stream still runs; it calls griddepcontrol.wait where it must not).
template <typename Kernel, typename... Args>
static cudaError_t launch_maybe_pdl(Kernel k, int grid, int threads, int smem, bool pdl, cudaStream_t s,
                                    Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, args...);
}

template <int D>
static cudaError_t launch_attn_d(const AttnParams& p, int grid, int W, bool pdl, cudaStream_t s) {
    const int smem = attn_smem_bytes<D>(W, p.G);
    auto k = p.o_fp32 ? attn_kernel<D, true> : attn_kernel<D, false>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = launch_maybe_pdl(k, grid, kAttnThreads, smem, pdl, s, p);
    if (e != cudaSuccess || p.n_split == 1) return e;
    const int rows = p.B * p.Hq;
    if (p.n_split <= kCombineWarpMaxSplits) {
        return launch_maybe_pdl(attn_combine_warp_kernel<D>, (rows + 7) / 8, 256, 0, pdl, s,
                                static_cast<const float*>(p.ws), p.O, p.o_fp32, rows, p.n_split);
    }
    return launch_maybe_pdl(attn_combine_cta_kernel<D>, rows, kCombineThreads, 0, pdl, s,
                            static_cast<const float*>(p.ws), p.O, p.o_fp32, p.n_split);
}

static dak_status launch_attn_kernels(const void* Q, const dak_placement* KV, const void* host_src,
                                      const int* seq_lens, int H_q, float scale, void* O, void* ws, size_t ws_bytes,
                                      const dak_tuning* t, cudaStream_t stream, int o_fp32, const LinkHandoff* link) {
    if (link && link->signals) *link->signals = 0;
    if (!KV || KV->kind != 1 || !Q || !O) return DAK_ERR_INVALID;
    if (H_q <= 0 || H_q % KV->H_kv) return DAK_ERR_INVALID;
    const int G = H_q / KV->H_kv;
    if (G > 16) return DAK_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(Q) & 15) || (reinterpret_cast<uintptr_t>(O) & 15)) return DAK_ERR_ALIGN;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DAK_ERR_CUDA;
    if (dev != KV->device) return DAK_ERR_INVALID;
    const int n_split = (t && t->n_split > 0) ? t->n_split : default_split(KV->B, KV->H_kv, KV->L);
    if (n_split > kMaxSplits) return DAK_ERR_INVALID;
    const size_t need = dak_attn_workspace_bytes(KV->B, H_q, KV->D, n_split);
    if (need > 0 && (!ws || ws_bytes < need)) return DAK_ERR_INVALID;
    if (need > 0 && (reinterpret_cast<uintptr_t>(ws) & 7)) return DAK_ERR_ALIGN;  // the combine reads float2
    if (KV->h_s > 0 && !host_src) return DAK_ERR_INVALID;

    AttnParams p{};
    p.Q = static_cast<const __nv_bfloat16*>(Q);
    p.kv[0] = static_cast<const uint8_t*>(host_src);
    p.kv[1] = static_cast<const uint8_t*>(KV->hbm_ptr);
    p.seq_lens = seq_lens;
    p.O = O;
    p.o_fp32 = o_fp32 ? 1 : 0;
    p.ws = static_cast<float*>(ws);
    p.B = KV->B;
    p.Hq = H_q;
    p.Hkv = KV->H_kv;
    p.G = G;
    p.L = KV->L;
    p.h_s = KV->h_s;
    p.n_split = n_split;
    p.split_len = ((KV->L + n_split - 1) / n_split + kChunkTok - 1) / kChunkTok * kChunkTok;
    const float sc = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(KV->D));
    p.scale_log2 = sc * 1.4426950408889634f;
    p.head_bytes = KV->head_bytes;
    p.st = status_ptr();
    if (!p.st) return DAK_ERR_CUDA;
    p.host_units = static_cast<long long>(KV->h_s) * n_split;
    p.hbm_units = (static_cast<long long>(KV->B) * KV->H_kv - KV->h_s) * n_split;
    const int host_units_i = static_cast<int>(std::min<long long>(p.host_units, 1 << 30));
    const int hbm_units_i = static_cast<int>(std::min<long long>(p.hbm_units, 1 << 30));
    int W_ring = (t && t->hbm_window > 0) ? std::min(t->hbm_window, kAttnMaxStages) : kAttnStages;
    if (!(t && t->hbm_window > 0) && p.host_units + p.hbm_units <= device_sm_count()) {
        // one CTA per SM holds every unit: a ring as deep as a unit's chunks (up to the
        // maximum) puts all of them in flight at once (1 request x 16 splits of 4K context:
        // 11.5 -> 10.8 us)
        W_ring = std::max(W_ring, std::min(p.split_len / kChunkTok, kAttnMaxStages));
    }
    if (t && t->window > 0) W_ring = std::max(W_ring, std::min(t->window, kAttnMaxStages));
    const int per_sm = KV->D == 128 ? attn_ctas_per_sm<128>(W_ring, G) : attn_ctas_per_sm<64>(W_ring, G);
    Sched sc2 = schedule(host_units_i, hbm_units_i, device_sm_count() * per_sm, t, kAttnDefaultHostCtas,
                         std::min(kAttnDefaultHostWindow, W_ring), W_ring, W_ring);
    p.n_host_ctas = sc2.n_host_ctas;
    p.n_hbm_ctas = sc2.n_hbm_ctas;
    p.host_window = sc2.host_window;
    p.hbm_window = sc2.hbm_window;
    const int grid = p.n_host_ctas + p.n_hbm_ctas;
    if (grid == 0) return DAK_OK;
    const int W = std::max(p.host_window, p.hbm_window);
    const bool pdl = t && t->pdl > 0;
    p.wait_newest = t && t->pdl == 2;
    if (link && link->ctr) {
        p.link = link->ctr;
        p.link_after = link->after;
    }
    cudaError_t e = KV->D == 128 ? launch_attn_d<128>(p, grid, W, pdl, stream) : launch_attn_d<64>(p, grid, W, pdl, stream);
    if (e == cudaSuccess && link && link->signals && p.link) *link->signals = p.n_host_ctas;
    return cuda_status(e);
}

dak_status launch_attn(const void* Q, const dak_placement* KV, const void* host_src, const int* seq_lens, int H_q,
                       float scale, void* O, void* ws, size_t ws_bytes, const dak_tuning* t, cudaStream_t stream,
                       int o_fp32, const LinkHandoff* link) {
    // a public launch that joins a handoff sequence (dak_link_begin, tuning link)
    LinkHandoff own;
    int own_signals = 0;
    const bool joined = !link && link_join(t, &own);
    if (joined) {
        own.signals = &own_signals;
        link = &own;
    }
    const dak_status r =
        launch_attn_kernels(Q, KV, host_src, seq_lens, H_q, scale, O, ws, ws_bytes, t, stream, o_fp32, link);
    if (joined && r == DAK_OK) link_commit(t, own_signals);
    return r;
}

}  // namespace dak

extern "C" size_t dak_attn_workspace_bytes(int B, int H_q, int D, int n_split) {
    if (B <= 0 || H_q <= 0 || D <= 0 || n_split <= 1) return 0;
    return static_cast<size_t>(B) * H_q * n_split * (D + 2) * sizeof(float);
}

extern "C" int dak_attn_default_split(const dak_placement* KV) {
    if (!KV || KV->kind != 1) return 0;
    return dak::default_split(KV->B, KV->H_kv, KV->L);
}

extern "C" dak_status dak_attn(const void* Q, const dak_placement* KV, const int* seq_lens, int H_q, float scale,
                               void* O, void* workspace, size_t ws_bytes, const dak_tuning* tuning, void* stream) {
    if (!KV) return DAK_ERR_INVALID;
    return dak::launch_attn(Q, KV, KV->host_dev, seq_lens, H_q, scale, O, workspace, ws_bytes, tuning,
                            static_cast<cudaStream_t>(stream));
}

extern "C" dak_status dak_attn_f32(const void* Q, const dak_placement* KV, const int* seq_lens, int H_q,
                                   float scale, void* O, void* workspace, size_t ws_bytes, const dak_tuning* tuning,
                                   void* stream) {
    if (!KV) return DAK_ERR_INVALID;
    return dak::launch_attn(Q, KV, KV->host_dev, seq_lens, H_q, scale, O, workspace, ws_bytes, tuning,
                            static_cast<cudaStream_t>(stream), 1);
}

extern "C" dak_status dak_attn_staged(const void* Q, const dak_placement* KV, const void* staging,
                                      const int* seq_lens, int H_q, float scale, void* O, void* workspace,
                                      size_t ws_bytes, const dak_tuning* tuning, void* stream) {
    if (!KV || (KV->h_s > 0 && !staging)) return DAK_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(staging) & 15) return DAK_ERR_ALIGN;
    return dak::launch_attn(Q, KV, staging, seq_lens, H_q, scale, O, workspace, ws_bytes, tuning,
                            static_cast<cudaStream_t>(stream));
}
