// SplitK_GEMM for decode: C = A x B where the tile rows of A are split between pinned,
// device-mapped host memory and HBM ("DAK: Direct-Access-Enabled GPU Memory Offloading
// with Optimal Efficiency for LLM Inference", section 4.1, Fig. 5).
//
// One persistent launch. CTAs [0, n_host) take the host tile rows, the others the HBM
// tile rows; a CTA never reads both tiers (section 4.1, "Kernel over Partitioned
// Memory"). Inside a CTA one producer thread streams m x kc chunks of its tile row into
// a ring of shared-memory slots with single bulk asynchronous copies (the copy engine of
// TMA) while other warps do the math (section 4.1, "Asynchronous TMA Access"). Host CTAs
// keep at most `host_window` chunks in flight: the static congestion window of section
// 4.3.1. Each tile row is read by exactly one CTA, which computes all N columns, so no
// host byte crosses the link twice (the locality half of section 4.3.2's scheduling).
//
// Placement layout of a tile row (both tiers): 64 rows x K_pad columns stored k-group
// major, [K_pad/8][64 rows][8 columns] bf16: every 8 x 8 block (8 rows x 16 bytes) is
// contiguous, every chunk of kc columns is one contiguous range, and that range is
// already the no-swizzle K-major operand layout the tcgen05 tensor cores read.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "dak_device.cuh"

namespace dak {

// Chunking of a CTA's ring. kcb == kc: each ring stage holds its A chunk (kc columns) and the
// matching B chunk. kcb < kc: the A ring holds kc-wide chunks only and B streams through its
// own ring of wb slots of kcb columns, kc / kcb of them per A chunk. Chunking never changes
// the sequence of K = 16 MMA steps, so it never changes a result.
struct Chunks {
    int kc, kcb;
    int stages, stage_bytes;       // A ring (stage = A chunk [+ B chunk when kcb == kc])
    int wb, b_ring_off, b_slot_bytes;
};

struct GemmParams {
    const uint8_t* a_host;  // tile rows 0 .. h-1 (device-visible address of the host mapping)
    const uint8_t* a_hbm;   // tile rows h .. T-1
    const __nv_bfloat16* B; // [N][K]
    void* C;                // [N][M]
    int M, K, K_pad, N, N_pad, T, h;
    int n_host_ctas, n_hbm_ctas, host_window, hbm_window;  // host/HBM counts are in clusters of S CTAs
    int c_fp32;
    long long tile_bytes;
    DevStatus* st;
    int b3d;      // B arrives in one 3-D tensor copy per stage (else several 2-D copies)
    int S;        // CTAs per cluster splitting each tile row's K range (1 = no split)
    int red_off;  // byte offset (from the aligned ring base) of the partial-sum area, S > 1
    int NC;       // CTAs per cluster sharing each tile row across 256-row blocks of B (1 = off)
    int glu;      // rows interleaved gate/up: C[n][row/2] = silu(gate) * up, C is [N][M/2]
    // Ring layout per role: ch[0] for CTAs reading HBM tiles, ch[1] for CTAs reading host
    // tiles (they differ only for wide B, where host tiles stream A in larger chunks)
    Chunks ch[2];
};

// SwiGLU of one gate / up pair (the same expression as the decoder's standalone kernel)
__device__ __forceinline__ float swiglu_pair(float g, float u) { return g / (1.f + expf(-g)) * u; }

// Tiles of this CTA: role, first tile, stride, count, and the chunk range [c_lo, c_hi) of
// every tile row that this CTA (rank `rank` of its cluster) accumulates.
struct TileIter {
    Chunks c;  // this CTA's ring layout
    bool host;
    int first, stride, count;
    const uint8_t* base;
    int window;
    int rank, c_lo, c_hi;
};

__device__ __forceinline__ TileIter tiles_of_cta(const GemmParams& p) {
    TileIter it;
    const int cl = p.S > 1 ? p.S : p.NC;  // CTAs per cluster
    const int b = blockIdx.x / cl;        // cluster index
    it.c = p.ch[b < p.n_host_ctas ? 1 : 0];
    const int nch = (p.K_pad + it.c.kc - 1) / it.c.kc;
    it.rank = cl > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    it.c_lo = p.S > 1 ? it.rank * nch / p.S : 0;
    it.c_hi = p.S > 1 ? (it.rank + 1) * nch / p.S : nch;
    if (b < p.n_host_ctas) {
        it.host = true;
        it.first = b;
        it.stride = p.n_host_ctas;
        it.count = (p.h > b) ? (p.h - b + p.n_host_ctas - 1) / p.n_host_ctas : 0;
        it.base = p.a_host;
        it.window = p.host_window;
    } else {
        int j = b - p.n_host_ctas;
        int nh = p.T - p.h;
        it.host = false;
        it.first = p.h + j;
        it.stride = p.n_hbm_ctas;
        it.count = (nh > j) ? (nh - j + p.n_hbm_ctas - 1) / p.n_hbm_ctas : 0;
        it.base = p.a_hbm;
        it.window = p.hbm_window;
    }
    return it;
}

__device__ __forceinline__ const uint8_t* tile_src(const GemmParams& p, const TileIter& it, int t) {
    int local = it.host ? t : t - p.h;
    return it.base + static_cast<long long>(local) * p.tile_bytes;
}

// error location codes (upper 32 bits of the status info)
enum : uint32_t {
    W_PROD_EMPTY = 1, W_CONS_FULL = 2, W_MMA_FULL = 3, W_MMA_ACC = 4, W_EPI_ACC = 5, W_DRAIN = 6, W_BPROD_EMPTY = 7,
    W_RED_FULL = 8, W_RED_EMPTY = 9, W_FWD_FULL = 10, W_FWD_PEER = 11, W_ARM_EMPTY = 12
};

// Wait (bounded, ignoring the abort flag) for the last fill of every ring slot, so that no
// bulk copy is still writing shared memory when the CTA exits.
__device__ __forceinline__ void drain_fills(uint64_t* full, int window, long long issued, DevStatus* st) {
    volatile int dummy = 0;
    for (int s = 0; s < window; ++s) {
        if (issued <= s) break;
        long long last = ((issued - 1 - s) / window) * window + s;  // last iteration that used slot s
        uint32_t parity = static_cast<uint32_t>((last / window) & 1);
        mbar_wait(&full[s], parity, &dummy, st, DAK_ERR_TIMEOUT, W_DRAIN);
    }
}

// ======================================================================================
// Loading B (the hidden states, shared by every CTA and L2-resident). Each stage's B chunk
// is one tensor-map copy issued by its own thread, so that the stream of A copies is never
// held up behind several smaller copies (on this GPU every bulk copy costs a CTA a fixed
// ~0.2-0.4 us, and a CTA's copies overlap only partly).
//   kUmmaB : 128-byte swizzled K-major blocks [kc/64][N_pad rows][64 columns] (the tcgen05
//            B operand); a 3-D box {64, N_pad, kc/64} when K % 64 == 0, else kc/64 2-D boxes.
//   kCoreB : plain blocks [kc/256][N rows][256 columns]; a 3-D box {256, N, kc/256} when
//            K % 256 == 0, else kc/256 2-D boxes.
// Columns past K and rows past N read as zero (tensor-map bounds fill).
// ======================================================================================
enum BKind { kCoreB = 0, kUmmaB = 1 };

__device__ __forceinline__ void issue_b(const GemmParams& p, const CUtensorMap* bmap, uint8_t* dst, int k0,
                                        uint64_t* bar, int kind, int row0, int kcb) {
    const int blk = kind == kUmmaB ? 64 : 256;
    const int rows = kind == kUmmaB ? p.N_pad : p.N;
    const int nblk = kcb / blk;
    if (p.b3d) {
        tma_load_3d(dst, bmap, 0, row0, k0 / blk, bar);
    } else {
        for (int b = 0; b < nblk; ++b) tma_load_2d(dst + b * rows * blk * 2, bmap, k0 + blk * b, row0, bar);
    }
}

__device__ __forceinline__ uint32_t b_stage_bytes(const GemmParams& p, int kind, int kcb) {
    return static_cast<uint32_t>(kcb) * 2u * static_cast<uint32_t>(kind == kUmmaB ? p.N_pad : p.N);
}

// Producer loops. `is_a` streams the tile rows of A (one bulk copy per stage), otherwise the
// matching chunk of B. Both wait for the slot to be released and then arm the stage's full
// barrier with their own byte count.
__device__ __forceinline__ void produce(const GemmParams& p, const TileIter& it, const CUtensorMap* bmap, uint8_t* smem,
                                        uint64_t* full, uint64_t* empty, volatile int* abort, bool is_a, int kind) {
    const int W = it.window;
    const uint64_t pol_a = policy_evict_first();
    // the weights never depend on the previous kernel of the stream; the hidden states may
    if (!is_a) grid_dep_wait();
    long long i = 0;
    for (int ti = 0; ti < it.count && !*abort; ++ti) {
        const int t = it.first + ti * it.stride;
        const uint8_t* src = tile_src(p, it, t);
        for (int c = it.c_lo; c < it.c_hi; ++c, ++i) {
            const int s = static_cast<int>(i % W);
            if (i >= W && !mbar_wait(&empty[s], static_cast<uint32_t>(((i / W) - 1) & 1), abort, p.st,
                                     DAK_ERR_TIMEOUT, is_a ? W_PROD_EMPTY : W_BPROD_EMPTY)) {
                goto done;
            }
            const int k0 = c * it.c.kc;
            uint8_t* dst = smem + static_cast<size_t>(s) * it.c.stage_bytes;
            if (is_a) {
                const uint32_t a_bytes = static_cast<uint32_t>(min(it.c.kc, p.K_pad - k0)) * 128u;
                mbar_arrive_expect_tx(&full[s], a_bytes);
                bulk_g2s(dst, src + static_cast<long long>(k0) * 128, a_bytes, &full[s], pol_a);
            } else {
                mbar_arrive_expect_tx(&full[s], b_stage_bytes(p, kind, it.c.kcb));
                issue_b(p, bmap, dst + it.c.kc * 128, k0, &full[s], kind, p.NC > 1 ? it.rank * p.N_pad : 0, it.c.kcb);
            }
        }
    }
done:
    drain_fills(full, W, i, p.st);
}

// B producer of the wide-B layout (kcb < kc): every A chunk's kc columns of B arrive as
// kc / kcb copies into B's own ring, each arming its slot's full barrier.
__device__ __forceinline__ void produce_b_ring(const GemmParams& p, const TileIter& it, const CUtensorMap* bmap,
                                               uint8_t* smem, uint64_t* b_full, uint64_t* b_empty,
                                               volatile int* abort) {
    grid_dep_wait();  // the hidden states may come from the previous kernel of the stream
    const int WB = it.c.wb;
    const int row0 = p.NC > 1 ? it.rank * p.N_pad : 0;
    long long ib = 0;
    for (int ti = 0; ti < it.count && !*abort; ++ti) {
        for (int c = it.c_lo; c < it.c_hi; ++c) {
            const int kce = min(it.c.kc, p.K_pad - c * it.c.kc);
            for (int sub = 0; sub * it.c.kcb < kce; ++sub, ++ib) {
                const int sb = static_cast<int>(ib % WB);
                if (ib >= WB && !mbar_wait(&b_empty[sb], static_cast<uint32_t>(((ib / WB) - 1) & 1), abort, p.st,
                                           DAK_ERR_TIMEOUT, W_BPROD_EMPTY)) {
                    goto done;
                }
                mbar_arrive_expect_tx(&b_full[sb], b_stage_bytes(p, kUmmaB, it.c.kcb));
                issue_b(p, bmap, smem + it.c.b_ring_off + static_cast<size_t>(sb) * it.c.b_slot_bytes,
                        c * it.c.kc + sub * it.c.kcb, &b_full[sb], kUmmaB, row0, it.c.kcb);
            }
        }
    }
done:
    drain_fills(b_full, WB, ib, p.st);
}

// Shared tile rows across the 256-row blocks of a wide B (NC > 1). Rank 0 of the cluster
// fetches every A chunk (host or HBM) once; its forwarder copies each arrived chunk from its
// ring slot into the same slot of every other rank with shared-to-shared bulk copies, waits
// until the copies have read the slot, and then releases it. The other ranks only arm their
// full barrier with the chunk's byte count and, once their MMAs have finished with a slot,
// tell rank 0 that it may be refilled. Each host byte therefore crosses the host link once
// however many 256-row blocks B has (no multicast is involved).
// Run by the whole forwarder warp of rank 0: lane r - 1 copies to rank r, so the copies to
// the NC - 1 other ranks are issued in parallel.
__device__ __forceinline__ void forward_a(const GemmParams& p, const TileIter& it, uint8_t* smem, uint64_t* full,
                                          uint64_t* empty, uint64_t* peer_empty, volatile int* abort) {
    const int W = it.window;
    const int lane = threadIdx.x & 31;
    const int r = lane + 1;  // the rank this lane forwards to
    long long i = 0;
    for (int ti = 0; ti < it.count; ++ti) {
        for (int c = it.c_lo; c < it.c_hi; ++c, ++i) {
            const int s = static_cast<int>(i % W);
            bool ok = mbar_wait(&full[s], static_cast<uint32_t>((i / W) & 1), abort, p.st, DAK_ERR_TIMEOUT, W_FWD_FULL);
            if (ok && i >= W)
                ok = mbar_wait_cluster(&peer_empty[s], static_cast<uint32_t>(((i / W) - 1) & 1), abort, p.st,
                                       DAK_ERR_TIMEOUT, W_FWD_PEER);
            if (!__all_sync(0xffffffffu, ok)) goto done;
            if (r < p.NC) {
                const int k0 = c * it.c.kc;
                const uint32_t a_bytes = static_cast<uint32_t>(min(it.c.kc, p.K_pad - k0)) * 128u;
                uint8_t* slot = smem + static_cast<size_t>(s) * it.c.stage_bytes;
                bulk_s2s_cluster(mapa_shared(smem_u32(slot), static_cast<uint32_t>(r)), slot, a_bytes,
                                 mapa_shared(smem_u32(&full[s]), static_cast<uint32_t>(r)));
                bulk_commit_group();
                bulk_wait_group_read0();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    }
done:
    if (r < p.NC) bulk_wait_group0();
    __syncwarp();
}

__device__ __forceinline__ void arm_forwarded_a(const GemmParams& p, const TileIter& it, uint64_t* full,
                                                uint64_t* empty, uint64_t* peer_empty, volatile int* abort) {
    const int W = it.window;
    long long i = 0;
    for (int ti = 0; ti < it.count && !*abort; ++ti) {
        for (int c = it.c_lo; c < it.c_hi; ++c, ++i) {
            const int s = static_cast<int>(i % W);
            if (i >= W) {
                if (!mbar_wait(&empty[s], static_cast<uint32_t>(((i / W) - 1) & 1), abort, p.st, DAK_ERR_TIMEOUT,
                               W_ARM_EMPTY))
                    goto done;
                mbar_arrive_remote(mapa_shared(smem_u32(&peer_empty[s]), 0));
            }
            const int k0 = c * it.c.kc;
            mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(min(it.c.kc, p.K_pad - k0)) * 128u);
        }
    }
done:
    drain_fills(full, W, i, p.st);
}

// ======================================================================================
// CUDA-core path, N in 1..7: warp-level FMA, fp32 accumulation, shuffle reduction.
// Warps: 0 = A producer, 1 = B producer, 2..9 = consumers (consumer w owns rows 8w .. 8w+7).
// ======================================================================================
constexpr int kCoreConsumers = 8;
constexpr int kCoreThreads = 32 * (2 + kCoreConsumers);

template <int N>
__global__ void __launch_bounds__(kCoreThreads, 1)
    gemm_core_kernel(const GemmParams p, const __grid_constant__ CUtensorMap bmap) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ uint64_t full[8], empty[8];
    __shared__ int abort_flag;
    volatile int* abort = &abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const TileIter it = tiles_of_cta(p);
    const int W = it.window;
    uint8_t* smem = smem_raw;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < W; ++s) {
            mbar_init(&full[s], 2);  // A producer + B producer
            mbar_init(&empty[s], kCoreConsumers);
        }
        fence_mbar_init();
        prefetch_tmap(&bmap);
    }
    __syncthreads();
    grid_dep_launch();

    if (warp < 2) {
        if (lane == 0) produce(p, it, &bmap, smem, full, empty, abort, warp == 0, kCoreB);
        return;
    }

    // consumers (C may be read by the previous kernel of the stream: wait before writing it)
    grid_dep_wait();
    const int w = warp - 2;       // row group 0..7
    const int r = lane & 7;       // row within the group
    const int kq = lane >> 3;     // k-group phase 0..3
    long long i = 0;
    for (int ti = 0; ti < it.count; ++ti) {
        const int t = it.first + ti * it.stride;
        float acc[N];
#pragma unroll
        for (int n = 0; n < N; ++n) acc[n] = 0.f;
        for (int c = it.c_lo; c < it.c_hi; ++c, ++i) {
            const int s = static_cast<int>(i % W);
            if (!mbar_wait(&full[s], static_cast<uint32_t>((i / W) & 1), abort, p.st, DAK_ERR_TIMEOUT, W_CONS_FULL)) {
                return;
            }
            const int k0 = c * it.c.kc;
            const int kgr = min(min(it.c.kc, p.K_pad - k0), p.K - k0) >> 3;  // real k-groups in this chunk
            const uint8_t* st = smem + static_cast<size_t>(s) * it.c.stage_bytes;
            const uint8_t* bst = st + it.c.kc * 128;
            for (int kg = kq; kg < kgr; kg += 4) {
                const uint4 a = *reinterpret_cast<const uint4*>(st + kg * 1024 + w * 128 + r * 16);
                const float a0 = bf_lo(a.x), a1 = bf_hi(a.x), a2 = bf_lo(a.y), a3 = bf_hi(a.y);
                const float a4 = bf_lo(a.z), a5 = bf_hi(a.z), a6 = bf_lo(a.w), a7 = bf_hi(a.w);
                // B block of 256 columns holding this k-group: [N rows][512 bytes]
                const uint8_t* bb = bst + (kg >> 5) * (N * 512) + (kg & 31) * 16;
#pragma unroll
                for (int n = 0; n < N; ++n) {
                    const uint4 b = *reinterpret_cast<const uint4*>(bb + n * 512);
                    float v = acc[n];
                    v = fmaf(a0, bf_lo(b.x), v);
                    v = fmaf(a1, bf_hi(b.x), v);
                    v = fmaf(a2, bf_lo(b.y), v);
                    v = fmaf(a3, bf_hi(b.y), v);
                    v = fmaf(a4, bf_lo(b.z), v);
                    v = fmaf(a5, bf_hi(b.z), v);
                    v = fmaf(a6, bf_lo(b.w), v);
                    v = fmaf(a7, bf_hi(b.w), v);
                    acc[n] = v;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        // reduce the four k phases: lanes r, r+8, r+16, r+24 hold the same row
#pragma unroll
        for (int n = 0; n < N; ++n) {
            float v = acc[n];
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            acc[n] = v;
        }
        const int row = t * kTileM + w * 8 + r;
        if (p.glu) {
            // rows 2j (gate) and 2j + 1 (up) are lanes r and r ^ 1 of this group
            float up[N];
#pragma unroll
            for (int n = 0; n < N; ++n) up[n] = __shfl_xor_sync(0xffffffffu, acc[n], 1);
            if (kq == 0 && row < p.M && !(row & 1)) {
                const int half = p.M >> 1, col = row >> 1;
#pragma unroll
                for (int n = 0; n < N; ++n) {
                    const float a = swiglu_pair(acc[n], up[n]);
                    if (p.c_fp32) {
                        reinterpret_cast<float*>(p.C)[static_cast<long long>(n) * half + col] = a;
                    } else {
                        reinterpret_cast<__nv_bfloat16*>(p.C)[static_cast<long long>(n) * half + col] =
                            __float2bfloat16_rn(a);
                    }
                }
            }
        } else if (kq == 0 && row < p.M) {
#pragma unroll
            for (int n = 0; n < N; ++n) {
                if (p.c_fp32) {
                    reinterpret_cast<float*>(p.C)[static_cast<long long>(n) * p.M + row] = acc[n];
                } else {
                    reinterpret_cast<__nv_bfloat16*>(p.C)[static_cast<long long>(n) * p.M + row] =
                        __float2bfloat16_rn(acc[n]);
                }
            }
        }
    }
}

// ======================================================================================
// Tensor-core path, N in 8..256: tcgen05.mma (M = 64 rows of A, N = N_pad hidden-state
// columns, K = 16 per instruction), fp32 accumulators in TMEM, double-buffered.
// Warps: 0 = A producer (bulk copies), 1 = TMEM allocator + MMA issuer,
//        2..5 = epilogue (TMEM -> registers -> C), 6 = B producer (tensor-map copies).
// ======================================================================================
constexpr int kUmmaThreads = 8 * 32;

// TMEM lane holding output row `row` (0..63) of an M = 64 accumulator: rows 16q .. 16q+15
// sit in lanes 32q .. 32q+15 of sub-partition q.
__device__ __forceinline__ int umma_m64_row_of_lane(int q, int lane) { return lane < 16 ? q * 16 + lane : -1; }

__global__ void __launch_bounds__(kUmmaThreads, 1)
    gemm_umma_kernel(const GemmParams p, const __grid_constant__ CUtensorMap bmap) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint64_t full[8], empty[8], acc_full[2], acc_empty[2];
    __shared__ uint64_t red_full, red_empty;  // cluster split: partials in / partial buffer free
    __shared__ uint64_t peer_empty[8];        // wide B, rank 0: every other rank has freed the slot
    __shared__ uint64_t b_full[8], b_empty[8];  // wide B: B's own ring
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;
    volatile int* abort = &abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const TileIter it = tiles_of_cta(p);
    const int W = it.window;
    // 1024-byte aligned ring (128-byte swizzle atoms must start on 1024-byte boundaries)
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int a_stage_bytes = it.c.kc * 128;
    const int bblk_bytes = p.N_pad * 128;  // one 64-column block of B
    uint32_t tmem_cols = 32;
    while (tmem_cols < static_cast<uint32_t>(2 * p.N_pad)) tmem_cols <<= 1;
    const uint32_t acc_stride = tmem_cols >> 1;  // column offset of the second accumulator

    if (threadIdx.x == 0) {
        abort_flag = 0;
        const bool fwd = p.NC > 1 && it.rank == 0;
        const bool b_ring = it.c.kcb < it.c.kc;
        for (int s = 0; s < W; ++s) {
            mbar_init(&full[s], b_ring ? 1 : 2);  // A producer (or A arming) [+ B producer]
            mbar_init(&empty[s], fwd ? 2 : 1);    // MMA commit (+ the forwarder on rank 0)
            if (fwd) mbar_init(&peer_empty[s], p.NC - 1);
        }
        if (b_ring) {
            for (int s = 0; s < it.c.wb; ++s) {
                mbar_init(&b_full[s], 1);
                mbar_init(&b_empty[s], 1);
            }
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        if (p.S > 1) {
            mbar_init(&red_full, (p.S - 1) * 128);  // every epilogue thread of every partner, per tile
            mbar_init(&red_empty, 128);             // every epilogue thread of the leader, per tile
        }
        fence_mbar_init();
        prefetch_tmap(&bmap);
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base_sh, tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (p.S > 1 || p.NC > 1) cluster_sync_all();  // partners' barriers exist before any remote access
    grid_dep_launch();
    const uint32_t tmem = tmem_base_sh;

    if (warp == 0 || warp == 6) {
        if (lane == 0) {
            if (warp == 0 && p.NC > 1 && it.rank > 0) {
                arm_forwarded_a(p, it, full, empty, peer_empty, abort);
            } else if (warp == 6 && it.c.kcb < it.c.kc) {
                produce_b_ring(p, it, &bmap, smem, b_full, b_empty, abort);
            } else {
                produce(p, it, &bmap, smem, full, empty, abort, warp == 0, kUmmaB);
            }
        }
    } else if (warp == 7) {
        if (p.NC > 1 && it.rank == 0) forward_a(p, it, smem, full, empty, peer_empty, abort);
    } else if (warp == 1) {
        // The whole warp runs the loop (so that loop state and descriptors stay warp-uniform);
        // one elected lane issues the MMAs and commits.
        const uint32_t idesc = idesc_bf16_f32(64, static_cast<uint32_t>(p.N_pad));
        const bool leader = elect_one();
        long long i = 0, ib = 0;
        uint64_t* last_bar = nullptr;
        uint32_t last_par = 0;
        for (int ti = 0; ti < it.count; ++ti) {
            const int ab = ti & 1;
            if (ti >= 2 && !mbar_wait(&acc_empty[ab], static_cast<uint32_t>(((ti >> 1) - 1) & 1), abort, p.st,
                                      DAK_ERR_TIMEOUT, W_MMA_ACC)) {
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + static_cast<uint32_t>(ab) * acc_stride;
            bool ok = true;
            for (int c = it.c_lo; c < it.c_hi; ++c, ++i) {
                const int s = static_cast<int>(i % W);
                // a forwarded A chunk is written by another CTA of the cluster
                const bool got = p.NC > 1 ? mbar_wait_cluster(&full[s], static_cast<uint32_t>((i / W) & 1), abort,
                                                              p.st, DAK_ERR_TIMEOUT, W_MMA_FULL)
                                          : mbar_wait(&full[s], static_cast<uint32_t>((i / W) & 1), abort, p.st,
                                                      DAK_ERR_TIMEOUT, W_MMA_FULL);
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int kce = min(it.c.kc, p.K_pad - c * it.c.kc);
                const uint32_t a_base = smem_u32(smem + static_cast<size_t>(s) * it.c.stage_bytes);
                // A: no swizzle, K-major; 8x8 blocks of one k-group are 128 B apart along M,
                // k-groups are 64 rows x 16 B = 1024 B apart along K (+2048 B per MMA).
                // B: 128-byte swizzle, K-major; 8-row groups 1024 B apart, 64-column blocks
                // N_pad x 128 B apart, +32 B per 16 columns inside a block.
                for (int sub = 0; sub * it.c.kcb < kce && ok; ++sub) {
                    uint32_t b_base = a_base + static_cast<uint32_t>(a_stage_bytes);
                    int sb = -1;
                    if (it.c.kcb < it.c.kc) {  // wide B: this sub-chunk's B comes from B's own ring
                        sb = static_cast<int>(ib % it.c.wb);
                        if (!mbar_wait(&b_full[sb], static_cast<uint32_t>((ib / it.c.wb) & 1), abort, p.st,
                                       DAK_ERR_TIMEOUT, W_MMA_FULL)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        b_base = smem_u32(smem + it.c.b_ring_off + static_cast<size_t>(sb) * it.c.b_slot_bytes);
                    }
                    const int k_sub = sub * it.c.kcb;
                    const int kcs = min(it.c.kcb, kce - k_sub);
                    const uint64_t ad0 = smem_desc(a_base + static_cast<uint32_t>((k_sub >> 3) * 1024), 1024u, 128u, 0u);
                    const uint64_t bd0 = smem_desc(b_base, 16u, 1024u, 2u);
                    if (leader) {
                        for (int kb = 0; kb < kcs; kb += 64) {
                            const uint64_t bdb = bd0 + (static_cast<uint64_t>((kb >> 6) * bblk_bytes) >> 4);
                            const uint64_t adb = ad0 + (static_cast<uint64_t>(kb >> 3) * 1024u >> 4);
                            const int nk = min(4, (kcs - kb) >> 4);
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                if (j < nk) {
                                    umma_bf16(d_tmem, adb + static_cast<uint64_t>(j * 128),
                                              bdb + static_cast<uint64_t>(j * 2), idesc,
                                              (c > it.c_lo || k_sub > 0 || kb > 0 || j > 0) ? 1u : 0u);
                                }
                            }
                        }
                        if (sb >= 0) umma_commit(&b_empty[sb]);
                    }
                    __syncwarp();
                    if (sb >= 0) {
                        ++ib;
                        last_bar = &b_empty[sb];
                        last_par = static_cast<uint32_t>(((ib - 1) / it.c.wb) & 1);
                    }
                }
                if (!ok) break;
                if (leader) umma_commit(&empty[s]);
                __syncwarp();
                last_bar = &empty[s];
                last_par = static_cast<uint32_t>((i / W) & 1);
            }
            if (!ok) break;
            if (leader) umma_commit(&acc_full[ab]);
            __syncwarp();
            last_bar = &acc_full[ab];
            last_par = static_cast<uint32_t>((ti >> 1) & 1);
        }
        if (last_bar) {  // every issued MMA has finished before TMEM is released
            volatile int dummy = 0;
            mbar_wait(last_bar, last_par, &dummy, p.st, DAK_ERR_TIMEOUT, W_DRAIN);
        }
        __syncwarp();
    } else {
        // epilogue warps 2..5 -> TMEM sub-partitions 2, 3, 0, 1. With a cluster split the
        // partners send their fp32 partial tiles into the leader's shared memory; the leader
        // adds them to its own in rank order (a fixed order, independent of the placement).
        const int q = warp & 3;
        const int row_in_tile = umma_m64_row_of_lane(q, lane);
        const bool leader = p.S > 1 ? it.rank == 0 : true;  // wide B: every rank writes its own rows
        const int n_off = p.NC > 1 ? it.rank * p.N_pad : 0;  // first hidden-state row of this CTA's block
        grid_dep_wait();  // C may be read by the previous kernel of the stream
        float* red = reinterpret_cast<float*>(smem + p.red_off);  // [S-1][64 rows][N_pad] on the leader
        for (int ti = 0; ti < it.count; ++ti) {
            const int ab = ti & 1;
            if (!mbar_wait(&acc_full[ab], static_cast<uint32_t>((ti >> 1) & 1), abort, p.st, DAK_ERR_TIMEOUT,
                           W_EPI_ACC)) {
                break;
            }
            tc_fence_after();
            const int t = it.first + ti * it.stride;
            const int row = t * kTileM + row_in_tile;
            const bool valid = row_in_tile >= 0 && row < p.M;
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(ab) * acc_stride;
            if (!leader) {
                // wait until the leader has consumed this CTA's previous partial
                if (ti > 0 && !mbar_wait_cluster(&red_empty, static_cast<uint32_t>((ti - 1) & 1), abort, p.st,
                                                 DAK_ERR_TIMEOUT, W_RED_EMPTY)) {
                    break;
                }
                const int r_own = row_in_tile >= 0 ? row_in_tile : 0;
                const uint32_t dst =
                    mapa_shared(smem_u32(red + static_cast<size_t>((it.rank - 1) * kTileM + r_own) * p.N_pad), 0);
                for (int n0 = 0; n0 < p.N_pad; n0 += 8) {
                    uint32_t v[8];
                    tmem_ld8(taddr + static_cast<uint32_t>(n0), v);
                    tmem_wait_ld();
                    if (row_in_tile >= 0) {
                        st_cluster_v4(dst + n0 * 4, __uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]),
                                      __uint_as_float(v[3]));
                        st_cluster_v4(dst + n0 * 4 + 16, __uint_as_float(v[4]), __uint_as_float(v[5]),
                                      __uint_as_float(v[6]), __uint_as_float(v[7]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[ab]);
                mbar_arrive_remote(mapa_shared(smem_u32(&red_full), 0));
                continue;
            }
            if (p.S > 1 && !mbar_wait_cluster(&red_full, static_cast<uint32_t>(ti & 1), abort, p.st, DAK_ERR_TIMEOUT,
                                              W_RED_FULL)) {
                break;
            }
            for (int n0 = 0; n0 < p.N_pad; n0 += 8) {
                uint32_t v[8];
                tmem_ld8(taddr + static_cast<uint32_t>(n0), v);
                tmem_wait_ld();
                float f[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) f[j] = __uint_as_float(v[j]);
                if (valid) {
                    for (int r = 1; r < p.S; ++r) {
                        const float4* pr = reinterpret_cast<const float4*>(
                            red + static_cast<size_t>((r - 1) * kTileM + row_in_tile) * p.N_pad + n0);
                        const float4 x0 = pr[0], x1 = pr[1];
                        f[0] += x0.x; f[1] += x0.y; f[2] += x0.z; f[3] += x0.w;
                        f[4] += x1.x; f[5] += x1.y; f[6] += x1.z; f[7] += x1.w;
                    }
                }
                if (p.glu) {
                    // rows 2j (gate) and 2j + 1 (up) sit in neighbouring lanes of this sub-partition
                    float up[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) up[j] = __shfl_xor_sync(0xffffffffu, f[j], 1);
                    if (valid && !(row_in_tile & 1)) {
                        const int half = p.M >> 1, col = row >> 1;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int n = n_off + n0 + j;
                            if (n < p.N) {
                                const float a = swiglu_pair(f[j], up[j]);
                                if (p.c_fp32) {
                                    reinterpret_cast<float*>(p.C)[static_cast<long long>(n) * half + col] = a;
                                } else {
                                    reinterpret_cast<__nv_bfloat16*>(p.C)[static_cast<long long>(n) * half + col] =
                                        __float2bfloat16_rn(a);
                                }
                            }
                        }
                    }
                } else if (valid) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int n = n_off + n0 + j;
                        if (n < p.N) {
                            if (p.c_fp32) {
                                reinterpret_cast<float*>(p.C)[static_cast<long long>(n) * p.M + row] = f[j];
                            } else {
                                reinterpret_cast<__nv_bfloat16*>(p.C)[static_cast<long long>(n) * p.M + row] =
                                    __float2bfloat16_rn(f[j]);
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[ab]);
            for (int r = 1; r < p.S; ++r) mbar_arrive_remote(mapa_shared(smem_u32(&red_empty), static_cast<uint32_t>(r)));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (p.S > 1 || p.NC > 1) cluster_sync_all();  // no CTA leaves while a partner may still touch its shared memory
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
}

// ======================================================================================
// host side
// ======================================================================================
using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
        }
    });
    return fn;
}

// Tensor map over B [N][K] for one kind of stage layout. Uses a single 3-D box per stage when
// K is a multiple of the block width (then every box element inside the map's bounds is an
// element of B); otherwise 2-D boxes. Sets *b3d accordingly.
static bool make_b_map(CUtensorMap* map, const void* B, int K, int N, int N_pad, int kc, int kind, int* b3d) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const int blk = kind == kUmmaB ? 64 : 256;
    const int rows = kind == kUmmaB ? N_pad : N;
    const CUtensorMapSwizzle swz = kind == kUmmaB ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
    if (K % blk == 0) {
        cuuint64_t dims[3] = {static_cast<cuuint64_t>(blk), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(K / blk)};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, static_cast<cuuint64_t>(blk) * 2};
        cuuint32_t box[3] = {static_cast<cuuint32_t>(blk), static_cast<cuuint32_t>(rows), static_cast<cuuint32_t>(kc / blk)};
        cuuint32_t estr[3] = {1, 1, 1};
        if (enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(B), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS) {
            *b3d = 1;
            return true;
        }
    }
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(blk), static_cast<cuuint32_t>(rows)};
    cuuint32_t estr[2] = {1, 1};
    *b3d = 0;
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(B), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kSmemBudget = 216 * 1024;           // one CTA per SM
constexpr int kSmemBudgetTwoPerSm = 108 * 1024;  // two CTAs per SM
constexpr int kDefaultHostCtas = 32;
constexpr int kMaxBlockN = 256;          // hidden-state rows of one CTA's tile
constexpr int kMaxWideN = 4 * kMaxBlockN;  // rows of one launch: a cluster of up to 4 CTAs shares A
constexpr int kDefaultHostWindow = 4;

// Launch with the optional cluster dimension and programmatic-dependent-launch attribute.
template <typename Kernel>
static cudaError_t launch_ex(Kernel k, int grid, int threads, int smem, int cluster, bool pdl, cudaStream_t s,
                             const GemmParams& p, const CUtensorMap& bmap) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = static_cast<unsigned>(n);
    return cudaLaunchKernelEx(&cfg, k, p, bmap);
}

// One launch over up to kMaxWideN hidden-state rows: one CTA per tile row up to 256 rows
// (the widest tcgen05 tile used here), a cluster of ceil(N / 256) CTAs per tile row beyond.
static dak_status launch_gemm_block(const dak_placement* A, const void* host_src, const void* B, void* C, int N,
                                    int c_fp32, const dak_tuning* t, cudaStream_t stream) {
    if (!A || A->kind != 0) return DAK_ERR_INVALID;
    if (N < 1 || N > kMaxWideN) return DAK_ERR_INVALID;
    if (A->M == 0 || A->T == 0) return DAK_OK;  // nothing to compute; C may be empty
    if (!B || !C) return DAK_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(B) & 15) || (reinterpret_cast<uintptr_t>(C) & 15)) return DAK_ERR_ALIGN;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DAK_ERR_CUDA;
    if (dev != A->device) return DAK_ERR_INVALID;

    GemmParams p{};
    p.a_host = static_cast<const uint8_t*>(host_src);
    p.a_hbm = static_cast<const uint8_t*>(A->hbm_ptr);
    p.B = static_cast<const __nv_bfloat16*>(B);
    p.C = C;
    p.M = static_cast<int>(A->M);
    p.K = static_cast<int>(A->K);
    p.K_pad = static_cast<int>(A->K_pad);
    p.N = N;
    // wide B: NC CTAs of a cluster share each tile row, CTA r computing rows [256 r, 256 r + 256)
    p.NC = N > kMaxBlockN ? (N + kMaxBlockN - 1) / kMaxBlockN : 1;
    p.N_pad = N > kMaxBlockN ? kMaxBlockN : (N + 7) & ~7;
    p.T = A->T;
    p.h = A->h;
    p.c_fp32 = c_fp32 ? 1 : 0;
    p.tile_bytes = A->tile_bytes;
    p.glu = A->glu;
    p.S = 1;
    p.st = status_ptr();
    if (!p.st) return DAK_ERR_CUDA;

    const bool umma = N >= 8;
    const int kind = umma ? kUmmaB : kCoreB;
    const int sms = device_sm_count();
    const int rows_b = umma ? p.N_pad : N;
    const int NC = p.NC;
    auto stage_of = [&](int k) { return (k * 128 + k * 2 * rows_b + 1023) & ~1023; };

    // Cluster split of each tile row's K range, chosen from the shape only (never from the
    // placement, so that results are bit-identical across offload ratios): when there are
    // fewer tile rows than SMs, S CTAs share a tile row and two CTAs run on each SM, which
    // multiplies the copy streams that keep HBM busy.
    auto red_of = [&](int s_) { return (s_ - 1) * kTileM * p.N_pad * 4; };
    // two stages of at least 128 columns beside the partial-sum area
    auto fits = [&](int s_, int budget_) { return 2 * stage_of(128) + red_of(s_) + 1024 <= budget_; };
    // CTAs of one cluster wait on each other, so they must never wait for TMEM: a split is
    // used only while two CTAs' accumulators (2 x 2 x N_pad columns) fit in one SM's TMEM.
    const bool can_split = umma && p.N_pad <= 128 && !(t && t->split_k == 1);
    int S = 1, per_sm = 1;
    if (can_split && (p.T < sms || (t && t->split_k > 1))) {
        const bool user = t && t->split_k > 1;
        // automatic: enough CTAs for two per SM, but each CTA still streams >= ~448 KiB of its
        // tile row (shorter slices are dominated by per-launch and pipeline-fill costs)
        const int by_bytes = static_cast<int>(p.tile_bytes / (448 * 1024));
        const int want = user ? std::min(8, t->split_k)
                              : std::max(1, std::min(8, std::min((2 * sms) / p.T, by_bytes)));
        if (fits(want, kSmemBudgetTwoPerSm)) {
            S = want;
            per_sm = want > 1 ? 2 : 1;
        } else {
            S = user ? want : std::max(1, std::min(8, sms / p.T));
            while (S > 1 && red_of(S) + 2 * stage_of(64) + 1024 > kSmemBudget) --S;
        }
    }
    if (umma && t && (t->ctas_per_sm == 1 || t->ctas_per_sm == 2)) per_sm = t->ctas_per_sm;
    const int budget = per_sm == 2 ? kSmemBudgetTwoPerSm : kSmemBudget;
    int kc;
    if (t && t->chunk_k > 0) {
        kc = t->chunk_k;
    } else if (!umma) {
        kc = 512;
    } else if (S > 1 || per_sm == 2) {
        // the widest chunk that leaves two stages beside the partial-sum area
        kc = 64;
        for (int cand : {512, 384, 256, 192, 128}) {
            if (2 * stage_of(cand) + red_of(S) + 1024 <= budget) {
                kc = cand;
                break;
            }
        }
    } else {
        // 64 KiB A copies where two such stages fit, 32 KiB otherwise
        kc = p.N_pad <= 32 ? 512 : (p.N_pad <= 64 ? 256 : (p.N_pad <= 128 ? 128 : 64));
    }
    if (kc % 64 != 0 || kc > 1024 || (!umma && kc % 256 != 0)) return DAK_ERR_INVALID;
    // Ring layouts. Shared tile rows (NC > 1): A in 256-column chunks and B through its own
    // ring of 64-column chunks, so that A copies and forwards stay large while B fills the
    // rest. One CTA per tile row with wide B (N_pad > 128): CTAs reading HBM keep the unified
    // ring, which keeps more B in flight; CTAs reading host tiles take the split layout, whose
    // 32 KiB A chunks keep more host bytes in flight (host reads are latency-bound).
    const bool b_ring_all = umma && NC > 1;
    const bool b_ring_host = umma && p.N_pad > 128 && !(t && t->chunk_k > 0);
    if (b_ring_all && !(t && t->chunk_k > 0)) kc = 256;
    const int nch = (p.K_pad + kc - 1) / kc;
    S = std::min(S, nch);
    if (S == 1) per_sm = 1;
    if (umma && t && (t->ctas_per_sm == 1 || t->ctas_per_sm == 2)) per_sm = t->ctas_per_sm;
    if (NC > 1) per_sm = 1;  // each CTA holds 2 x 256 TMEM columns, the whole TMEM of an SM
    p.S = S;
    const int CL = S > 1 ? S : NC;  // CTAs per cluster
    const int red_bytes = S > 1 ? red_of(S) : 0;
    const int ring_budget = per_sm == 2 ? kSmemBudgetTwoPerSm : kSmemBudget;
    auto layout = [&](int kc_, bool split, Chunks* L) -> bool {
        L->kc = kc_;
        L->kcb = split ? 64 : kc_;
        if (split) {
            L->stage_bytes = (kc_ * 128 + 1023) & ~1023;
            L->b_slot_bytes = (p.N_pad * L->kcb * 2 + 1023) & ~1023;
            const int avail = ring_budget - red_bytes - 1024;
            L->stages = std::min(4, std::max(2, avail / 2 / L->stage_bytes));  // about half for A
            L->wb = std::min(8, (avail - L->stages * L->stage_bytes) / L->b_slot_bytes);
            if (L->wb < 2) {
                L->stages = 2;
                L->wb = std::min(8, (avail - L->stages * L->stage_bytes) / L->b_slot_bytes);
            }
            if (L->wb < 2) return false;
        } else {
            L->stage_bytes = stage_of(kc_);
            L->stages = std::min(8, (ring_budget - red_bytes - (umma ? 1024 : 0)) / L->stage_bytes);
            L->wb = 0;
            L->b_slot_bytes = 0;
            if (L->stages < 1 || (L->stages < 2 && !(t && t->chunk_k > 0))) return false;
        }
        L->b_ring_off = L->stages * L->stage_bytes;
        return true;
    };
    if (!layout(kc, b_ring_all, &p.ch[0])) return DAK_ERR_INVALID;
    p.ch[1] = p.ch[0];
    if (!b_ring_all && b_ring_host && S == 1 && p.h > 0) {
        if (!layout(256, true, &p.ch[1])) p.ch[1] = p.ch[0];
    }
    if (p.ch[0].kcb != p.ch[1].kcb) return DAK_ERR_INVALID;  // one B tensor map serves both
    const int kcb = p.ch[0].kcb;
    auto ring_bytes = [](const Chunks& L) { return L.stages * L.stage_bytes + L.wb * L.b_slot_bytes; };
    const int rings = std::max(ring_bytes(p.ch[0]), ring_bytes(p.ch[1]));
    p.red_off = rings;
    const int smem = rings + red_bytes + (umma ? 1024 : 0);
    const int max_stages = std::max(p.ch[0].stages, p.ch[1].stages);

    // schedule in cluster units
    dak_tuning tc{};
    if (t) tc = *t;
    tc.host_ctas = std::max(1, (tc.host_ctas > 0 ? tc.host_ctas : kDefaultHostCtas) / CL);
    if (tc.hbm_ctas > 0) tc.hbm_ctas = std::max(1, tc.hbm_ctas / CL);
    Sched sc = schedule(p.h, p.T - p.h, std::max(1, (sms * per_sm) / CL), &tc, std::max(1, kDefaultHostCtas / CL),
                        std::min(kDefaultHostWindow, p.ch[1].stages), p.ch[0].stages, max_stages);
    p.n_host_ctas = sc.n_host_ctas;
    p.n_hbm_ctas = sc.n_hbm_ctas;
    p.host_window = std::min(sc.host_window, p.ch[1].stages);
    p.hbm_window = std::min(sc.hbm_window, p.ch[0].stages);
    const int grid = (p.n_host_ctas + p.n_hbm_ctas) * CL;
    if (grid == 0) return DAK_OK;
    if (p.h > 0 && !p.a_host) return DAK_ERR_INVALID;

    alignas(64) CUtensorMap bmap;
    int b3d = 0;
    if (!make_b_map(&bmap, B, p.K, N, p.N_pad, kcb, kind, &b3d)) return DAK_ERR_CUDA;
    p.b3d = b3d;

    const bool pdl = t && t->pdl > 0;
    cudaError_t e;
    if (umma) {
        e = launch_ex(gemm_umma_kernel, grid, kUmmaThreads, smem, CL, pdl, stream, p, bmap);
    } else {
        switch (N) {
            case 1: e = launch_ex(gemm_core_kernel<1>, grid, kCoreThreads, smem, 1, pdl, stream, p, bmap); break;
            case 2: e = launch_ex(gemm_core_kernel<2>, grid, kCoreThreads, smem, 1, pdl, stream, p, bmap); break;
            case 3: e = launch_ex(gemm_core_kernel<3>, grid, kCoreThreads, smem, 1, pdl, stream, p, bmap); break;
            case 4: e = launch_ex(gemm_core_kernel<4>, grid, kCoreThreads, smem, 1, pdl, stream, p, bmap); break;
            case 5: e = launch_ex(gemm_core_kernel<5>, grid, kCoreThreads, smem, 1, pdl, stream, p, bmap); break;
            case 6: e = launch_ex(gemm_core_kernel<6>, grid, kCoreThreads, smem, 1, pdl, stream, p, bmap); break;
            default: e = launch_ex(gemm_core_kernel<7>, grid, kCoreThreads, smem, 1, pdl, stream, p, bmap); break;
        }
    }
    return cuda_status(e);
}

// Any N, in column blocks of hidden-state rows (B rows and C rows of a block are
// contiguous), one launch each: by default blocks of up to kMaxWideN rows in which a
// cluster of ceil(rows / 256) CTAs shares each tile row, so the host tiles cross the link
// once per block; with column_blocks, blocks of 256 rows that each read the host tiles
// again. Clusters stop at 4 CTAs: forwarding every A chunk to 7 peers measured slower than
// two launches of 1024 rows.
dak_status launch_gemm(const dak_placement* A, const void* host_src, const void* B, void* C, int N, int c_fp32,
                       const dak_tuning* t, cudaStream_t stream) {
    if (!A || A->kind != 0) return DAK_ERR_INVALID;
    const int block = (t && t->column_blocks == 1) ? kMaxBlockN : kMaxWideN;
    if (N <= block) return launch_gemm_block(A, host_src, B, C, N, c_fp32, t, stream);
    if (!B || !C) return DAK_ERR_INVALID;
    const size_t b_row = static_cast<size_t>(A->K) * 2;
    const size_t c_row = static_cast<size_t>(A->glu ? A->M / 2 : A->M) * (c_fp32 ? 4 : 2);
    for (int n0 = 0; n0 < N; n0 += block) {
        const int nb = std::min(block, N - n0);
        const dak_status r = launch_gemm_block(A, host_src, static_cast<const uint8_t*>(B) + n0 * b_row,
                                               static_cast<uint8_t*>(C) + n0 * c_row, nb, c_fp32, t, stream);
        if (r != DAK_OK) return r;
    }
    return DAK_OK;
}

}  // namespace dak

extern "C" dak_status dak_gemm(const dak_placement* A, const void* B, void* C, int N, int c_fp32,
                               const dak_tuning* tuning, void* stream) {
    if (!A) return DAK_ERR_INVALID;
    return dak::launch_gemm(A, A->host_dev, B, C, N, c_fp32, tuning, static_cast<cudaStream_t>(stream));
}

extern "C" dak_status dak_gemm_staged(const dak_placement* A, const void* staging, const void* B, void* C, int N,
                                      int c_fp32, const dak_tuning* tuning, void* stream) {
    if (!A || (A->h > 0 && !staging)) return DAK_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(staging) & 15) return DAK_ERR_ALIGN;
    return dak::launch_gemm(A, staging, B, C, N, c_fp32, tuning, static_cast<cudaStream_t>(stream));
}
