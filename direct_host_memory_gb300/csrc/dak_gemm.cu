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
// 4.3.1. Each byte of a tile row is read by exactly one CTA, which computes all N columns
// for it, so no host byte crosses the link twice (the locality half of section 4.3.2's
// scheduling). A tile row's K range may be cut into P pieces, each a unit of work of its
// tier's CTAs, so that the units spread evenly over the SMs; the CTA that finishes a tile
// row's last piece adds the fp32 partial tiles in piece order.
//
// Placement layout (both tiers): the tier's tile rows in blocks of two, tier-local tile
// rows 2b and 2b + 1 stored together k-group major, [K_pad/8][128 rows][8 columns] bf16,
// 2b tile rows into the tier; with an odd count the last tile row is a block of its own,
// [K_pad/8][64][8]. Every 8 x 8 block (8 rows x 16 bytes) is contiguous, every chunk of kc
// columns of a block is one contiguous range, and that range is already the no-swizzle
// K-major operand layout the tcgen05 tensor cores read: a block of two is one M = 128
// operand, so one MMA covers 128 rows (twice the rows per instruction and per byte of B of
// an M = 64 tile row).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

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
    int a_cb;                      // bytes of A per column in a stage: 128 (one tile row) or 256 (two)
};

struct GemmParams {
    const uint8_t* a_host;  // tile rows 0 .. h-1 (device-visible address of the host mapping)
    const uint8_t* a_hbm;   // tile rows h .. T-1
    const __nv_bfloat16* B; // [N][K]
    void* C;                // [N][M]
    int M, K, K_pad, N, N_pad, T, h;
    int pairs;    // 1: a placement of 128-row tiles: every unit is a block of two tile rows (M = 128 MMAs)
    int hb, gb;   // blocks of the host tier and of the HBM tier (tile rows, or pairs of them)
    int n_host_ctas, n_hbm_ctas, host_window, hbm_window;  // host/HBM counts are in clusters of NC CTAs
    int c_fp32;
    long long tile_bytes;
    DevStatus* st;
    int b3d;      // B arrives in one 3-D tensor copy per stage (else several 2-D copies)
    int P;        // pieces per tile row: its K range is cut into P parts, each a unit of work
    int pstep;    // piece boundaries fall on multiples of this many columns (a B block: 64, 256)
    float* part;  // P > 1: fp32 partials, per block [P][64 or 128 rows][N_pad] (host blocks first)
    int* cnt;     // P > 1: per block, pieces finished so far (back to 0 after the last)
    int NC;       // CTAs per cluster sharing each tile row across 256-row blocks of B (1 = off)
    int glu;      // rows interleaved gate/up: C[n][row/2] = silu(gate) * up, C is [N][M/2]
    // Ring layout per role: ch[0] for CTAs reading HBM tiles, ch[1] for CTAs reading host
    // tiles (they differ only for wide B, where host tiles stream A in larger chunks)
    Chunks ch[2];
    // A decode step's RMSNorm folded into the GEMMs around it (see GemmFuse; null = off)
    float* res_x;
    const __nv_bfloat16* res_g;
    float* ss_out;
    const float* ss_in;
    int ss_tiles;
    float ss_inv_d, ss_eps;
    // host-link handoff of a decode step (link_wait / link_signal; null = off)
    unsigned* link;
    unsigned link_after;
};

// Fused RMSNorm (the decode step's norms folded into the GEMMs around them):
//  - a producer GEMM (res_x set) does not output its product: it adds it to the fp32 residual
//    stream, x[n][row] += acc, stores h[n][row] = bf16(x[n][row] * g[row]) as C (bf16), and
//    for every tile row t the sums of x^2 over the tile's 64 rows, ss_out[t][n];
//  - a consumer GEMM (ss_in set) multiplies hidden-state row n's accumulators by
//    r_n = 1 / sqrt(sum_t ss_in[t][n] / d + eps) before storing them (before SwiGLU).
// So consumer(h) = RMSNorm(x) * g . A^T with the 1 / rms factor applied after the product.
constexpr int kFuseMaxN = 128;  // hidden-state rows of a fused launch (one CTA per tile row)
constexpr int kFusePreloadN = 16;  // up to this many rows, the producer preloads x into registers

// SwiGLU of one gate / up pair (the same expression as the decoder's standalone kernel)
__device__ __forceinline__ float swiglu_pair(float g, float u) { return g / (1.f + expf(-g)) * u; }

// Blocks of a tier of n tile rows: one tile row each, or (pairs) n / 2 blocks of two and one of
// one when n is odd.
__host__ __device__ __forceinline__ int blocks_of(int n, int pairs) { return pairs ? (n + 1) / 2 : n; }

// Units of work of this CTA. A role's units are its blocks times P pieces (unit u is piece
// u % P of the role's block u / P); the CTA takes units first, first + stride, ... (count
// of them), so that the pieces of one block go to different CTAs.
struct TileIter {
    Chunks c;  // this CTA's ring layout
    bool host;
    int tile0;  // first tile row of the role
    int first, stride, count;
    const uint8_t* base;
    int window;
    int rank;  // rank in the cluster of a wide B (0 otherwise)
};

__device__ __forceinline__ TileIter tiles_of_cta(const GemmParams& p, int cta = -1) {
    TileIter it;
    const int b = (cta < 0 ? static_cast<int>(blockIdx.x) : cta) / p.NC;  // cluster index
    it.c = p.ch[b < p.n_host_ctas ? 1 : 0];
    it.rank = p.NC > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    if (b < p.n_host_ctas) {
        const int units = p.hb * p.P;
        it.host = true;
        it.tile0 = 0;
        it.first = b;
        it.stride = p.n_host_ctas;
        it.count = (units > b) ? (units - b + p.n_host_ctas - 1) / p.n_host_ctas : 0;
        it.base = p.a_host;
        it.window = p.host_window;
    } else {
        const int j = b - p.n_host_ctas;
        const int units = p.gb * p.P;
        it.host = false;
        it.tile0 = p.h;
        it.first = j;
        it.stride = p.n_hbm_ctas;
        it.count = (units > j) ? (units - j + p.n_hbm_ctas - 1) / p.n_hbm_ctas : 0;
        it.base = p.a_hbm;
        it.window = p.hbm_window;
    }
    return it;
}

// The ui-th unit of a CTA: a block (its first tile row t, whether it holds two tile rows)
// and its K range [k0, k1). A block's K range is cut into P pieces at multiples of pstep
// columns (one block of the B layout, so that every chunk starts on one), from the shape only.
struct Piece {
    int t;      // first tile row of the block (global)
    int lb;     // block index within the tier
    int blk;    // block index over both tiers (host blocks first): the piece counter's index
    int m128;   // a pair block (M = 128: rows 0..63 tile row t, 64..127 tile row t + 1)
    int pair;   // m128 and tile row t + 1 holds rows of A (a 128-row tile may end past M)
    long long prow;  // first row of the block's partials in the split workspace (x P x N_pad floats)
    int idx, k0, k1;
};

// PM: the tile height fixed at compile time (0: 64 rows, 1: 128) in a kernel instantiated
// per height, or -1: the launch's p.pairs
template <int PM = -1>
__device__ __forceinline__ Piece piece_of(const GemmParams& p, const TileIter& it, int ui) {
    const int u = it.first + ui * it.stride;
    Piece q;
    q.lb = u / p.P;
    q.idx = u % p.P;
    const int n_tier = it.host ? p.h : p.T - p.h;
    q.m128 = PM < 0 ? p.pairs : PM;
    q.t = it.tile0 + (q.m128 ? 2 * q.lb : q.lb);
    q.pair = (q.m128 && 2 * q.lb + 1 < n_tier && (q.t + 1) * kTileM < p.M) ? 1 : 0;
    q.blk = (it.host ? 0 : p.hb) + q.lb;
    q.prow = static_cast<long long>(q.blk) * (q.m128 ? 2 * kTileM : kTileM);
    const int steps = (p.K_pad + p.pstep - 1) / p.pstep;
    q.k0 = (q.idx * steps / p.P) * p.pstep;
    q.k1 = min(((q.idx + 1) * steps / p.P) * p.pstep, p.K_pad);
    return q;
}

// rows of a block's partials, and where piece r's partial block starts
__device__ __forceinline__ int block_rows(const Piece& q) { return q.m128 ? 2 * kTileM : kTileM; }
__device__ __forceinline__ float* piece_part(const GemmParams& p, const Piece& q, int r) {
    return p.part + (q.prow * p.P + static_cast<long long>(r) * block_rows(q)) * p.N_pad;
}

// the block's bytes in its tier ([K_pad / 8][64 or 128 rows][8])
__device__ __forceinline__ const uint8_t* block_src(const GemmParams& p, const TileIter& it, const Piece& q) {
    return it.base + static_cast<long long>(q.m128 ? 2 * q.lb : q.lb) * p.tile_bytes;
}

// bytes of one column of a block's A, in the placement and in a stage
__device__ __forceinline__ int col_bytes(const Piece& q) { return q.m128 ? 256 : 128; }

// error location codes (upper 32 bits of the status info)
enum : uint32_t {
    W_PROD_EMPTY = 1, W_CONS_FULL = 2, W_MMA_FULL = 3, W_MMA_ACC = 4, W_EPI_ACC = 5, W_DRAIN = 6, W_BPROD_EMPTY = 7,
    W_FWD_FULL = 10, W_FWD_PEER = 11, W_ARM_EMPTY = 12, W_FIN_DONE = 13, W_FIN_FREED = 14
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

// Producer loops. `is_a` streams the blocks of A (one bulk copy per stage), otherwise the
// matching chunk of B. Both wait for the slot to be released and then arm the stage's full
// barrier with their own byte count. A stage holds A (kc x a_cb bytes), then B.
__device__ __forceinline__ void produce(const GemmParams& p, const TileIter& it, const CUtensorMap* bmap,
                                        uint8_t* smem, uint64_t* full, uint64_t* empty, volatile int* abort, bool is_a,
                                        int kind) {
    const int W = it.window;
    const uint64_t pol_a = policy_evict_first();
    // the weights never depend on the previous kernel of the stream; the hidden states may
    if (!is_a) grid_dep_wait();
    const bool link = is_a && it.host && p.link;
    if (link) link_wait(p.link, p.link_after, p.st);
    long long i = 0;
    for (int ui = 0; ui < it.count && !*abort; ++ui) {
        const Piece q = piece_of(p, it, ui);
        const uint8_t* src = block_src(p, it, q);
        for (int k0 = q.k0; k0 < q.k1; k0 += it.c.kc, ++i) {
            const int s = static_cast<int>(i % W);
            if (i >= W && !mbar_wait(&empty[s], static_cast<uint32_t>(((i / W) - 1) & 1), abort, p.st,
                                     DAK_ERR_TIMEOUT, is_a ? W_PROD_EMPTY : W_BPROD_EMPTY)) {
                goto done;
            }
            uint8_t* dst = smem + static_cast<size_t>(s) * it.c.stage_bytes;
            const int kce = min(it.c.kc, q.k1 - k0);
            if (is_a) {
                const int cb = col_bytes(q);
                const uint32_t a_bytes = static_cast<uint32_t>(kce * cb);
                mbar_arrive_expect_tx(&full[s], a_bytes);
                bulk_g2s(dst, src + static_cast<long long>(k0) * cb, a_bytes, &full[s], pol_a);
            } else {
                mbar_arrive_expect_tx(&full[s], b_stage_bytes(p, kind, it.c.kcb));
                issue_b(p, bmap, dst + it.c.kc * it.c.a_cb, k0, &full[s], kind, p.NC > 1 ? it.rank * p.N_pad : 0,
                        it.c.kcb);
            }
        }
    }
done:
    if (link) link_signal(p.link);
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
    for (int ui = 0; ui < it.count && !*abort; ++ui) {
        const Piece q = piece_of(p, it, ui);
        for (int k0 = q.k0; k0 < q.k1; k0 += it.c.kc) {
            const int kce = min(it.c.kc, q.k1 - k0);
            for (int sub = 0; sub * it.c.kcb < kce; ++sub, ++ib) {
                const int sb = static_cast<int>(ib % WB);
                if (ib >= WB && !mbar_wait(&b_empty[sb], static_cast<uint32_t>(((ib / WB) - 1) & 1), abort, p.st,
                                           DAK_ERR_TIMEOUT, W_BPROD_EMPTY)) {
                    goto done;
                }
                mbar_arrive_expect_tx(&b_full[sb], b_stage_bytes(p, kUmmaB, it.c.kcb));
                issue_b(p, bmap, smem + it.c.b_ring_off + static_cast<size_t>(sb) * it.c.b_slot_bytes,
                        k0 + sub * it.c.kcb, &b_full[sb], kUmmaB, row0, it.c.kcb);
            }
        }
    }
done:
    drain_fills(b_full, WB, ib, p.st);
}

// Shared tile rows across the 256-row blocks of a wide B (NC > 1). For host tile rows, rank 0
// of the cluster fetches every A chunk once; its forwarder copies each arrived chunk from its
// ring slot into the same slot of every other rank with shared-to-shared bulk copies, waits
// until the copies have read the slot, and then releases it. The other ranks only arm their
// full barrier with the chunk's byte count and, once their MMAs have finished with a slot,
// tell rank 0 that it may be refilled. Each host byte therefore crosses the host link once
// however many 256-row blocks B has (no multicast is involved). HBM tile rows are not
// forwarded: every rank streams its chunks itself, and since the ranks of a cluster read the
// same tile row together, L2 serves the repeats (HBM reads stay at one per byte; forwarding
// them to three peers made 4-CTA clusters 2.4x slower per tile row than 2-CTA ones).
// Run by the whole forwarder warp of rank 0: lane r - 1 copies to rank r, so the copies to
// the NC - 1 other ranks are issued in parallel.
__device__ __forceinline__ void forward_a(const GemmParams& p, const TileIter& it, uint8_t* smem, uint64_t* full,
                                          uint64_t* empty, uint64_t* peer_empty, volatile int* abort) {
    const int W = it.window;
    const int lane = threadIdx.x & 31;
    const int r = lane + 1;  // the rank this lane forwards to
    long long i = 0;
    for (int ui = 0; ui < it.count; ++ui) {
        const Piece q = piece_of(p, it, ui);
        for (int k0 = q.k0; k0 < q.k1; k0 += it.c.kc, ++i) {
            const int s = static_cast<int>(i % W);
            bool ok = mbar_wait(&full[s], static_cast<uint32_t>((i / W) & 1), abort, p.st, DAK_ERR_TIMEOUT, W_FWD_FULL);
            if (ok && i >= W)
                ok = mbar_wait_cluster(&peer_empty[s], static_cast<uint32_t>(((i / W) - 1) & 1), abort, p.st,
                                       DAK_ERR_TIMEOUT, W_FWD_PEER);
            if (!__all_sync(0xffffffffu, ok)) goto done;
            if (r < p.NC) {
                const uint32_t a_bytes = static_cast<uint32_t>(min(it.c.kc, q.k1 - k0) * col_bytes(q));
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
    for (int ui = 0; ui < it.count && !*abort; ++ui) {
        const Piece q = piece_of(p, it, ui);
        for (int k0 = q.k0; k0 < q.k1; k0 += it.c.kc, ++i) {
            const int s = static_cast<int>(i % W);
            if (i >= W) {
                if (!mbar_wait(&empty[s], static_cast<uint32_t>(((i / W) - 1) & 1), abort, p.st, DAK_ERR_TIMEOUT,
                               W_ARM_EMPTY))
                    goto done;
                mbar_arrive_remote(mapa_shared(smem_u32(&peer_empty[s]), 0));
            }
            mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(min(it.c.kc, q.k1 - k0) * col_bytes(q)));
        }
    }
done:
    drain_fills(full, W, i, p.st);
}

// ======================================================================================
// CUDA-core path, N = 1 (a GEMV): warp-level FMA, fp32 accumulation, shuffle reduction.
// Warps: 0 = A producer, 1 = B producer, 2..9 = consumers (consumer w owns rows 8w .. 8w+7),
// 10 = finisher of split tile rows (blocks of one tile row: the piece counter's index and the
// partials' position are the tile row's). With P > 1 the consumers store each piece's partial
// rows and move on; the finisher counts the piece in (one acquire-release atomic per piece) and,
// for a tile row's last piece, adds the P partials in piece order and writes C, so the
// count's round trip never stalls the FMA stream.
// ======================================================================================
constexpr int kCoreConsumers = 8;
constexpr int kCoreThreads = 32 * (3 + kCoreConsumers);
constexpr int kCoreDone = 4;  // units a finisher may lag behind the consumers

// GPU-scope atomic add with acquire and release semantics; returns the old value.
__device__ __forceinline__ int atomic_add_acq_rel(int* addr, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
    return old;
}

// C[n][row] for n < N of one output row (fp32 or bf16). With a SwiGLU placement, rows 2j
// (gate) and 2j + 1 (up) are held by lanes l and l ^ 1; the even lane writes C[n][j] =
// silu(gate) * up (C has M / 2 columns). Every lane of the warp calls this. Folded norm:
// fr scales acc[n] by rsc[n] first; fx adds acc to the residual (xpre / gpre: x[n][row] and
// g[row], preloaded) and writes C = bf16(x * g), returning x^2 in sq (0 elsewhere).
template <int N>
__device__ __forceinline__ void store_row(const GemmParams& p, float (&acc)[N], int row, bool write, bool fx,
                                          bool fr, const float (&rsc)[N], float (&sq)[N], const float (&xpre)[N],
                                          float gpre) {
#pragma unroll
    for (int n = 0; n < N; ++n) {
        if (fr) acc[n] *= rsc[n];
        sq[n] = 0.f;
    }
    if (p.glu) {
        float up[N];
#pragma unroll
        for (int n = 0; n < N; ++n) up[n] = __shfl_xor_sync(0xffffffffu, acc[n], 1);
        if (write && row < p.M && !(row & 1)) {
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
    } else if (fx) {
        if (write && row < p.M) {
            const float g = gpre;  // preloaded with x: xpre[n] = x[n][row], gpre = g[row]
#pragma unroll
            for (int n = 0; n < N; ++n) {
                const long long i = static_cast<long long>(n) * p.M + row;
                const float xn = xpre[n] + acc[n];
                p.res_x[i] = xn;
                reinterpret_cast<__nv_bfloat16*>(p.C)[i] = __float2bfloat16_rn(xn * g);
                sq[n] = xn * xn;
            }
        }
    } else if (write && row < p.M) {
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

// Fused norm, producer: x[n][row] (n < N) and g[row] of one output row, loaded ahead of the
// row's accumulators (x is written only by the epilogue that finishes the row's tile row).
template <int N>
__device__ __forceinline__ void preload_residual(const GemmParams& p, bool fx, int row, float (&xpre)[N],
                                                 float& gpre) {
    const bool ok = fx && row < p.M;
#pragma unroll
    for (int n = 0; n < N; ++n) xpre[n] = ok ? p.res_x[static_cast<long long>(n) * p.M + row] : 0.f;
    gpre = ok ? __bfloat162float(p.res_g[row]) : 0.f;
}

// Butterfly sum over the 32 lanes of a warp (every lane gets the total, in a fixed order).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// r_n of a consumer GEMM computed by one warp: lane l sums tile rows l, l + 32, ... in order,
// then the butterfly (the GEMV path's order; the tensor-core path has its own, fixed too).
template <int N>
__device__ __forceinline__ void warp_row_scales(const GemmParams& p, bool fr, int lane, float (&rsc)[N]) {
#pragma unroll
    for (int n = 0; n < N; ++n) {
        float v = 0.f;
        if (fr) {
            for (int t = lane; t < p.ss_tiles; t += 32) v += p.ss_in[static_cast<long long>(t) * p.N + n];
        }
        rsc[n] = rsqrtf(warp_sum(v) * p.ss_inv_d + p.ss_eps);
    }
}

// The 256 threads of the eight FMA warps meet (named barrier 2).
__device__ __forceinline__ void consumer_bar_sync() { asm volatile("bar.sync 2, 256;" ::: "memory"); }

// PAIRS: the placement's tiles are 128 rows (blocks of two tile rows); a separate
// instantiation, so that the 64-row path keeps its single-row inner loop.
template <int N, bool F, bool PAIRS>
__global__ void __launch_bounds__(kCoreThreads, 1)
    gemm_core_kernel(const GemmParams p, const __grid_constant__ CUtensorMap bmap) {
    // the folded norm's code exists only in the F = true instantiation
    const bool fx = F && p.res_x != nullptr;
    const bool fr = F && p.ss_in != nullptr;
    extern __shared__ __align__(1024) uint8_t smem_raw[];  // one declaration for both GEMM kernels
    __shared__ uint64_t full[8], empty[8];
    __shared__ uint64_t done[kCoreDone], freed[kCoreDone];  // split: partial rows stored / finisher done
    __shared__ float ssw[kCoreConsumers][N];                // fused norm: each consumer warp's 8 rows
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
        for (int j = 0; j < kCoreDone; ++j) {
            mbar_init(&done[j], kCoreConsumers);
            mbar_init(&freed[j], 1);
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
    if (warp == 2 + kCoreConsumers) {
        if (p.P == 1) return;
        // finisher: lane l sums rows l, l + 32 (, l + 64, l + 96 for a block of two tile rows)
        // of a block whose last piece this CTA ran
        grid_dep_wait();  // the split workspace may still be in use by the previous kernel
        float rsc[N];
        warp_row_scales<N>(p, fr, lane, rsc);
        for (int ui = 0; ui < it.count; ++ui) {
            const int j = ui % kCoreDone;
            if (!mbar_wait(&done[j], static_cast<uint32_t>((ui / kCoreDone) & 1), abort, p.st, DAK_ERR_TIMEOUT,
                           W_FIN_DONE)) {
                return;
            }
            const Piece pc = piece_of<PAIRS ? 1 : 0>(p, it, ui);
            const int nr = pc.pair ? 4 : 2;  // 32-row groups of the block
            float xp[4][N], gp[4];
            for (int g = 0; g < nr; ++g) preload_residual<N>(p, fx, pc.t * kTileM + lane + 32 * g, xp[g], gp[g]);
            int last = 0;
            if (lane == 0) {
                __threadfence();
                last = atomic_add_acq_rel(p.cnt + pc.blk, 1) + 1 == p.P;
                if (last) p.cnt[pc.blk] = 0;  // ready for the next launch
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            __syncwarp();
            if (last) {
                const float* src = piece_part(p, pc, 0);
                const long long blk_floats = static_cast<long long>(block_rows(pc)) * p.N_pad;
                float ssl[2][N];
#pragma unroll
                for (int n = 0; n < N; ++n) ssl[0][n] = ssl[1][n] = 0.f;
                for (int g = 0; g < nr; ++g) {
                    const int rr = lane + 32 * g;
                    float acc[N], sq[N];
#pragma unroll
                    for (int n = 0; n < N; ++n) {
                        float v = __ldcg(src + rr * p.N_pad + n);
                        for (int r = 1; r < p.P; ++r) v += __ldcg(src + r * blk_floats + rr * p.N_pad + n);
                        acc[n] = v;
                    }
                    store_row<N>(p, acc, pc.t * kTileM + rr, true, fx, fr, rsc, sq, xp[g], gp[g]);
#pragma unroll
                    for (int n = 0; n < N; ++n) ssl[g >> 1][n] += sq[n];
                }
                if (fx) {
                    for (int h = 0; h < (pc.pair ? 2 : 1); ++h) {
#pragma unroll
                        for (int n = 0; n < N; ++n) {
                            const float tot = warp_sum(ssl[h][n]);
                            if (lane == 0) p.ss_out[static_cast<long long>(pc.t + h) * p.N + n] = tot;
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&freed[j]);
        }
        return;
    }

    // consumers (C may be read by the previous kernel of the stream: wait before writing it)
    grid_dep_wait();
    float rsc[N];
    warp_row_scales<N>(p, fr, lane, rsc);
    const int w = warp - 2;       // row group 0..7 (of each tile row of the block)
    const int r = lane & 7;       // row within the group
    const int kq = lane >> 3;     // k-group phase 0..3
    long long i = 0;
    // after a wait that ran out, a fused launch's consumers skip the work but keep meeting
    // their named barrier, so that no warp is left waiting for one that gave up
    bool failed = false;
    for (int ui = 0; ui < it.count; ++ui) {
        const Piece q = piece_of<PAIRS ? 1 : 0>(p, it, ui);
        const int t = q.t;
        constexpr int kH = PAIRS ? 2 : 1;
        const int halves = (PAIRS && q.pair) ? 2 : 1;    // tile rows of the block that hold rows of A
        constexpr int kg_bytes = PAIRS ? 2048 : 1024;  // one k-group of the block in the stage
        float acc[kH][N], xp[kH][N], gp[kH];
#pragma unroll
        for (int h = 0; h < kH; ++h) gp[h] = 0.f;
        if (p.P == 1) {
#pragma unroll
            for (int h = 0; h < kH; ++h)
                if (h < halves) preload_residual<N>(p, fx, (t + h) * kTileM + w * 8 + r, xp[h], gp[h]);
        }
#pragma unroll
        for (int h = 0; h < kH; ++h)
#pragma unroll
            for (int n = 0; n < N; ++n) acc[h][n] = 0.f;
        for (int k0 = q.k0; k0 < q.k1 && !failed; k0 += it.c.kc, ++i) {
            const int s = static_cast<int>(i % W);
            if (!mbar_wait(&full[s], static_cast<uint32_t>((i / W) & 1), abort, p.st, DAK_ERR_TIMEOUT, W_CONS_FULL)) {
                if (!(fx && p.P == 1)) return;
                failed = true;
                break;
            }
            const int kgr = min(min(it.c.kc, q.k1 - k0), p.K - k0) >> 3;  // real k-groups in this chunk
            const uint8_t* st = smem + static_cast<size_t>(s) * it.c.stage_bytes;
            const uint8_t* bst = st + it.c.kc * it.c.a_cb;
            for (int kg = kq; kg < kgr; kg += 4) {
                // B block of 256 columns holding this k-group: [N rows][512 bytes]
                const uint8_t* bb = bst + (kg >> 5) * (N * 512) + (kg & 31) * 16;
#pragma unroll
                for (int h = 0; h < kH; ++h) {
                    if (h >= halves) break;
                    const uint4 a = *reinterpret_cast<const uint4*>(st + kg * kg_bytes + h * 1024 + w * 128 + r * 16);
                    const float a0 = bf_lo(a.x), a1 = bf_hi(a.x), a2 = bf_lo(a.y), a3 = bf_hi(a.y);
                    const float a4 = bf_lo(a.z), a5 = bf_hi(a.z), a6 = bf_lo(a.w), a7 = bf_hi(a.w);
#pragma unroll
                    for (int n = 0; n < N; ++n) {
                        const uint4 b = *reinterpret_cast<const uint4*>(bb + n * 512);
                        float v = acc[h][n];
                        v = fmaf(a0, bf_lo(b.x), v);
                        v = fmaf(a1, bf_hi(b.x), v);
                        v = fmaf(a2, bf_lo(b.y), v);
                        v = fmaf(a3, bf_hi(b.y), v);
                        v = fmaf(a4, bf_lo(b.z), v);
                        v = fmaf(a5, bf_hi(b.z), v);
                        v = fmaf(a6, bf_lo(b.w), v);
                        v = fmaf(a7, bf_hi(b.w), v);
                        acc[h][n] = v;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        // reduce the four k phases: lanes r, r+8, r+16, r+24 hold the same row
#pragma unroll
        for (int h = 0; h < kH; ++h) {
#pragma unroll
            for (int n = 0; n < N; ++n) {
                float v = acc[h][n];
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                acc[h][n] = v;
            }
        }
        if (p.P == 1) {
#pragma unroll
            for (int h = 0; h < kH; ++h) {
                if (h >= halves) break;
                float sq[N];
                store_row<N>(p, acc[h], (t + h) * kTileM + w * 8 + r, kq == 0 && !failed, fx, fr, rsc, sq, xp[h], gp[h]);
                if (fx) {
                    // the tile row's sums of x^2: each warp's 8 rows, then the 8 warps in order
#pragma unroll
                    for (int n = 0; n < N; ++n) {
                        const float v = warp_sum(sq[n]);
                        if (lane == 0) ssw[w][n] = v;
                    }
                    consumer_bar_sync();
                    if (w == 0 && lane < N) {
                        float tot = 0.f;
#pragma unroll
                        for (int ww = 0; ww < kCoreConsumers; ++ww) tot += ssw[ww][lane];
                        p.ss_out[static_cast<long long>(t + h) * p.N + lane] = tot;
                    }
                    consumer_bar_sync();  // ssw is rewritten by the next tile row
                }
            }
            continue;
        }
        // split block: this unit's partial rows to the workspace, then tell the finisher
        if (kq == 0) {
#pragma unroll
            for (int h = 0; h < kH; ++h) {
                if (h >= halves) break;
                float* mine = piece_part(p, q, q.idx) + (h * kTileM + w * 8 + r) * p.N_pad;
#pragma unroll
                for (int n = 0; n < N; ++n) mine[n] = acc[h][n];
            }
        }
        __syncwarp();
        const int j = ui % kCoreDone;
        if (ui >= kCoreDone && !mbar_wait(&freed[j], static_cast<uint32_t>(((ui / kCoreDone) - 1) & 1), abort, p.st,
                                          DAK_ERR_TIMEOUT, W_FIN_FREED)) {
            return;
        }
        if (lane == 0) mbar_arrive(&done[j]);
    }
}

// ======================================================================================
// Tensor-core path, N >= 2: tcgen05.mma (M = 64 rows of A for a single-row block, 128 for a
// pair block; N = N_pad <= 256 hidden-state columns; K = 16 per instruction), fp32
// accumulators in TMEM, double-buffered (one per unit of work, so the epilogue of one unit
// overlaps the MMAs of the next). Pair blocks (placements of 128-row tiles) give one MMA
// the work of two: at N_pad >= 128 a tile row is tensor-bound, and an M = 128 instruction
// keeps the tensor pipe only about 1.25x as long as an M = 64 one.
// Warps: 0 = A producer (bulk copies), 1 = TMEM allocator + MMA issuer,
//        2..5 = epilogue (TMEM -> registers -> C, or -> partial tile and the piece count),
//        6 = B producer (tensor-map copies), 7 = A forwarder of a wide-B cluster (NC > 1).
// ======================================================================================
constexpr int kUmmaThreads = 8 * 32;

// The n MMAs (K = 16 each) of one sub-chunk. Step m reads A two k-groups of the no-swizzle
// layout further on (a_step16 descriptor units: 2048 bytes for a 64-row operand, 4096 for a
// 128-row one) and B 32 bytes further inside a 64-column block, with one block (bblk16
// descriptor units) per 64 columns. The first step of a piece starts the
// accumulator; the rest go out four per asm block with 32-bit adds on the descriptors' low
// words (the start-address field, which never carries into the high word here).
__device__ __forceinline__ void issue_mmas(uint32_t d_tmem, uint64_t ad0, uint64_t bd0, uint32_t bblk16, int n,
                                           uint32_t idesc, bool accumulate, uint32_t a_step16) {
    const uint32_t a_lo = static_cast<uint32_t>(ad0), a_hi = static_cast<uint32_t>(ad0 >> 32);
    const uint32_t b_lo = static_cast<uint32_t>(bd0), b_hi = static_cast<uint32_t>(bd0 >> 32);
    auto a_at = [&](int m) { return a_lo + static_cast<uint32_t>(m) * a_step16; };
    auto b_at = [&](int m) { return b_lo + static_cast<uint32_t>(m >> 2) * bblk16 + static_cast<uint32_t>(m & 3) * 2u; };
    int m = 0;
    if (!accumulate && n > 0) {
        umma_bf16(d_tmem, ad0, bd0, idesc, 0u);
        m = 1;
    }
    for (; m + 4 <= n; m += 4) {
        umma_bf16_x4(d_tmem, a_at(m), a_at(m + 1), a_at(m + 2), a_at(m + 3), a_hi, b_at(m), b_at(m + 1), b_at(m + 2),
                     b_at(m + 3), b_hi, idesc);
    }
    for (; m < n; ++m) {
        umma_bf16(d_tmem, (static_cast<uint64_t>(a_hi) << 32) | a_at(m), (static_cast<uint64_t>(b_hi) << 32) | b_at(m),
                  idesc, 1u);
    }
}

constexpr int kMaxPieces = 8;       // pieces per tile row
constexpr int kMinPieceSteps = 8;   // 64-column steps of an automatically chosen piece

// C[n][row] for the 8 hidden-state rows n_base .. n_base + 7 of one output row (n < N only),
// fp32 or bf16. With a SwiGLU placement, rows 2j (gate) and 2j + 1 (up) are held by lanes l
// and l ^ 1: the even lane writes C[n][j] = silu(gate) * up (C has M / 2 columns). Every lane
// of the warp calls this (the pairing is a shuffle).
// Folded norm: fr scales f[j] by rsc[n_base + j] first; fx adds f to the residual (x read
// here or preloaded in xpre / gpre) and writes C = bf16(x * g), returning x^2 in sq.
__device__ __forceinline__ void store_c(const GemmParams& p, float (&f)[8], int row, bool valid, int n_base,
                                        bool fx, bool fr, const float* rsc, float (&sq)[8],
                                        const float* xpre = nullptr, float gpre = 0.f) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (fr && n_base + j < p.N) f[j] *= rsc[n_base + j];
        sq[j] = 0.f;
    }
    if (p.glu) {
        float up[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) up[j] = __shfl_xor_sync(0xffffffffu, f[j], 1);
        if (valid && !(row & 1)) {
            const int half = p.M >> 1, col = row >> 1;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int n = n_base + j;
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
    } else if (fx) {
        if (valid) {
            // x and g come preloaded (xpre: this block's 8 values) or are read here
            const float g = xpre ? gpre : __bfloat162float(p.res_g[row]);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int n = n_base + j;
                if (n < p.N) {
                    const long long i = static_cast<long long>(n) * p.M + row;
                    const float xn = (xpre ? xpre[j] : p.res_x[i]) + f[j];
                    p.res_x[i] = xn;
                    reinterpret_cast<__nv_bfloat16*>(p.C)[i] = __float2bfloat16_rn(xn * g);
                    sq[j] = xn * xn;
                }
            }
        }
    } else if (valid) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int n = n_base + j;
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

// The 128 threads of the four epilogue warps meet (named barrier 1; barrier 0 is __syncthreads).
__device__ __forceinline__ void epilogue_bar_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// TMEM lane holding output row `row` (0..63) of an M = 64 accumulator: rows 16q .. 16q+15
// sit in lanes 32q .. 32q+15 of sub-partition q.
__device__ __forceinline__ int umma_m64_row_of_lane(int q, int lane) { return lane < 16 ? q * 16 + lane : -1; }

// Fused norm, producer: the tile row's sums of x^2 per hidden-state row from the warps'
// partial sums (slots slot0 .. slot0 + slots - 1 in order), written by thread e = n. Every
// epilogue thread calls this.
__device__ __forceinline__ void fuse_tile_sums(const GemmParams& p, const float (*ssw)[kFuseMaxN], int t, int e,
                                               int slot0, int slots) {
    epilogue_bar_sync();  // every warp's sums are in
    if (e < p.N) {
        float v = 0.f;
        for (int k = slot0; k < slot0 + slots; ++k) v += ssw[k][e];
        p.ss_out[static_cast<long long>(t) * p.N + e] = v;
    }
    epilogue_bar_sync();  // the slots are rewritten by the next tile row
}

// Fused norm, producer: the tile rows' sums of x^2 of a unit's block (a pair block: rows
// 0..63 in slots 0, 1, rows 64..127 in slots 2, 3; a single-row block: slots 0 .. slots - 1).
__device__ __forceinline__ void fuse_block_sums(const GemmParams& p, const float (*ssw)[kFuseMaxN], const Piece& pc,
                                                int e, int single_slots) {
    if (pc.m128) {
        fuse_tile_sums(p, ssw, pc.t, e, 0, 2);
        if (pc.pair) fuse_tile_sums(p, ssw, pc.t + 1, e, 2, 2);
    } else {
        fuse_tile_sums(p, ssw, pc.t, e, 0, single_slots);
    }
}

// The output row (within its block) that TMEM lane `lane` of sub-partition qp holds: a pair
// block (M = 128) has rows 32 qp .. 32 qp + 31, a single-row block (M = 64) rows 16 qp ..
// 16 qp + 15 in lanes 0..15 (-1 elsewhere).
__device__ __forceinline__ int block_row_of_lane(bool m128, int qp, int lane) {
    return m128 ? qp * 32 + lane : umma_m64_row_of_lane(qp, lane);
}

// Whether row r of a block is an output row of this unit: rows 64..127 of a pair block only
// when its second tile row is in the tier, and never past M.
__device__ __forceinline__ bool block_row_ok(const GemmParams& p, const Piece& pc, int r) {
    return r >= 0 && (r < kTileM || pc.pair) && pc.t * kTileM + r < p.M;
}

// Fused norm, producer, up to 16 hidden-state rows: the residual values an epilogue thread
// adds to and the gain, loaded before the accumulator is ready (a round trip to L2 off the
// unit's tail); x is written only by the epilogue that finishes a block. In the split path
// thread e holds row e of a pair block (every column), or row e % 64 of a single-row block
// and the 8 columns from 8 (e / 64); in the one-piece path the row of its TMEM lane (rib) and
// every column.
__device__ __forceinline__ void preload_x(const GemmParams& p, const Piece& pc, int e, int rib,
                                          float (&xpre)[kFusePreloadN], float& gpre) {
    const bool split = p.P > 1;
    const int r = split ? (pc.m128 ? e : (e & 63)) : rib;
    const int xrow = pc.t * kTileM + r;
    const int xn0 = (split && !pc.m128) ? 8 * (e >> 6) : 0;
    const int xcols = (split && !pc.m128) ? 8 : p.N_pad;
    const bool ok = block_row_ok(p, pc, r);
#pragma unroll
    for (int j = 0; j < kFusePreloadN; ++j) {
        const int n = xn0 + j;
        const bool use = ok && j < xcols && n < p.N;
        xpre[j] = use ? p.res_x[static_cast<long long>(n) * p.M + xrow] : 0.f;
    }
    gpre = ok ? __bfloat162float(p.res_g[xrow]) : 0.f;
}

// One unit's epilogue, run by the four epilogue warps (thread e = 0..127; warp `warp` reads
// TMEM sub-partition warp & 3). A split block (P > 1): the CTA of every piece stores its fp32
// partial block in the workspace and counts the piece in; the CTA that counts the last one
// adds the P partials in piece order (a fixed order, whichever CTA ran which piece and
// whatever the placement) and writes C. No CTA waits for another. After a wait that ran
// out (`failed`), the threads skip the work but meet the epilogue's named barriers.
__device__ __forceinline__ void epilogue_unit(const GemmParams& p, const Piece& pc, uint32_t taddr, bool failed,
                                              uint64_t* acc_empty_ab, int warp, int lane, int e, int n_off, bool fx,
                                              bool fr, const float* rsc, float (*fuse_ssw)[kFuseMaxN],
                                              volatile int* last_piece, bool xpre_on,
                                              const float (&xpre)[kFusePreloadN], float gpre) {
    const int qp = warp & 3;
    const int rib = block_row_of_lane(pc.m128, qp, lane);
    const int row = pc.t * kTileM + rib;
    const bool valid = block_row_ok(p, pc, rib);
    const int blk_floats = block_rows(pc) * p.N_pad;  // one piece's partial block in the workspace
    if (p.P > 1) {
        float* mine = piece_part(p, pc, pc.idx);
        for (int n0 = 0; n0 < p.N_pad && !failed; n0 += 8) {
            uint32_t v[8];
            tmem_ld8(taddr + static_cast<uint32_t>(n0), v);
            tmem_wait_ld();
            if (rib >= 0) {  // (rows past the tier or M too: the sum skips them)
                float4* d = reinterpret_cast<float4*>(mine + rib * p.N_pad + n0);
                d[0] = make_float4(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]),
                                   __uint_as_float(v[3]));
                d[1] = make_float4(__uint_as_float(v[4]), __uint_as_float(v[5]), __uint_as_float(v[6]),
                                   __uint_as_float(v[7]));
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !failed) mbar_arrive(acc_empty_ab);  // the accumulator is free again
        // One thread counts the piece in, with release semantics for the 128 threads' stores
        // (ordered before it by the barrier) and acquire semantics for the other pieces'
        // partials, which the last piece's CTA reads next.
        epilogue_bar_sync();
        if (warp == 2 && lane == 0) {
            *last_piece = 0;
            if (!failed) {
                const int done = atomic_add_acq_rel(p.cnt + pc.blk, 1) + 1;
                *last_piece = done == p.P;
                if (done == p.P) p.cnt[pc.blk] = 0;  // ready for the next launch
            }
        }
        epilogue_bar_sync();
        if (!*last_piece) return;
        // The P partials, added in piece order. All 128 threads share the work: thread e takes
        // row e of a pair block (every 8-column block), or row e % 64 of a single-row block and
        // the 8-column blocks e / 64, e / 64 + 2, ...; lanes e and e ^ 1 hold rows 2j and 2j + 1
        // (the gate / up pair of a SwiGLU placement).
        const int rr = pc.m128 ? e : (e & 63);
        const int b0 = pc.m128 ? 0 : (e >> 6), bstep = pc.m128 ? 1 : 2;
        const int rrow = pc.t * kTileM + rr;
        const bool rok = block_row_ok(p, pc, rr);
        const float* src0 = piece_part(p, pc, 0) + rr * p.N_pad;
        for (int blk = b0; blk * 8 < p.N_pad; blk += bstep) {
            const float* src = src0 + blk * 8;
            float f[8];
            for (int r0 = 0; r0 < p.P; r0 += 4) {  // four partials in flight at a time
                float4 x[8];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    if (r0 + r < p.P) {
                        x[2 * r] = __ldcg(reinterpret_cast<const float4*>(src + (r0 + r) * blk_floats));
                        x[2 * r + 1] = __ldcg(reinterpret_cast<const float4*>(src + (r0 + r) * blk_floats + 4));
                    }
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    if (r0 + r == 0) {
                        f[0] = x[0].x; f[1] = x[0].y; f[2] = x[0].z; f[3] = x[0].w;
                        f[4] = x[1].x; f[5] = x[1].y; f[6] = x[1].z; f[7] = x[1].w;
                    } else if (r0 + r < p.P) {
                        f[0] += x[2 * r].x; f[1] += x[2 * r].y; f[2] += x[2 * r].z; f[3] += x[2 * r].w;
                        f[4] += x[2 * r + 1].x; f[5] += x[2 * r + 1].y; f[6] += x[2 * r + 1].z;
                        f[7] += x[2 * r + 1].w;
                    }
                }
            }
            float sq[8], xb[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) xb[j] = (pc.m128 && blk == 1) ? xpre[8 + j] : xpre[j];  // registers
            store_c(p, f, rrow, rok, n_off + blk * 8, fx, fr, rsc, sq, xpre_on ? xb : nullptr, gpre);
            if (fx) {
                // rows 32 w2 .. 32 w2 + 31 of the thread's warp w2 = e / 32: one sum per column
                // (a pair block: slot w2; a single-row block: slot w2 % 2, the column blocks of
                // the two halves being different)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float v = warp_sum(sq[j]);
                    if (lane == 0) fuse_ssw[pc.m128 ? (e >> 5) : ((e >> 5) & 1)][blk * 8 + j] = v;
                }
            }
        }
        if (fx) fuse_block_sums(p, fuse_ssw, pc, e, 2);
        return;
    }
    for (int n0 = 0; n0 < p.N_pad; n0 += 8) {
        float f[8];
        if (!failed) {
            uint32_t v[8];
            tmem_ld8(taddr + static_cast<uint32_t>(n0), v);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = __uint_as_float(v[j]);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = 0.f;
        }
        float sq[8], xb[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) xb[j] = n0 == 0 ? xpre[j] : xpre[8 + j];  // registers, not a stack copy
        store_c(p, f, row, valid && !failed, n_off + n0, fx, fr, rsc, sq, xpre_on ? xb : nullptr, gpre);
        if (fx) {
            // the rows of this warp's sub-partition: one sum per column
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float v = warp_sum(sq[j]);
                if (lane == 0) fuse_ssw[qp][n0 + j] = v;
            }
        }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0 && !failed) mbar_arrive(acc_empty_ab);
    if (fx) fuse_block_sums(p, fuse_ssw, pc, e, 4);
}

// PAIRS: the placement's tiles are 128 rows (an instantiation per height)
template <bool F, bool PAIRS>
__global__ void __launch_bounds__(kUmmaThreads, 1)
    gemm_umma_kernel(const GemmParams p, const __grid_constant__ CUtensorMap bmap,
                     const __grid_constant__ CUtensorMap bmap_host) {
    // the folded norm's code exists only in the F = true instantiation
    const bool fx = F && p.res_x != nullptr;
    const bool fr = F && p.ss_in != nullptr;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint64_t full[8], empty[8], acc_full[2], acc_empty[2];
    __shared__ uint64_t peer_empty[8];        // wide B, rank 0: every other rank has freed the slot
    __shared__ uint64_t b_full[8], b_empty[8];  // wide B: B's own ring
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;
    __shared__ int last_piece;  // split tile rows: this CTA finished the tile row's last piece
    __shared__ float fuse_ssw[4][kFuseMaxN];  // fused norm, producer: each warp's partial sums of x^2
    __shared__ float fuse_red[kFuseMaxN];     // fused norm, consumer: groups' partial sums
    __shared__ float fuse_r[kFuseMaxN];       // fused norm, consumer: r_n
    volatile int* abort = &abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const TileIter it = tiles_of_cta(p);
    const int W = it.window;
    // 1024-byte aligned ring (128-byte swizzle atoms must start on 1024-byte boundaries)
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int a_stage_bytes = it.c.kc * it.c.a_cb;  // A of the stage (128 or 256 bytes per column)
    const int bblk_bytes = p.N_pad * 128;     // one 64-column block of B
    uint32_t tmem_cols = 32;
    while (tmem_cols < static_cast<uint32_t>(2 * p.N_pad)) tmem_cols <<= 1;
    const uint32_t acc_stride = tmem_cols >> 1;  // column offset of the second accumulator

    if (threadIdx.x == 0) {
        abort_flag = 0;
        // host tiles in a cluster: rank 0 fetches and forwards (each host byte crosses the link
        // once); HBM tiles: every rank fetches its chunks itself (the cluster's ranks read the same
        // tile row together, so L2 serves the repeats)
        const bool fwd = p.NC > 1 && it.rank == 0 && it.host;
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
        fence_mbar_init();
        prefetch_tmap(&bmap);
        prefetch_tmap(&bmap_host);
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base_sh, tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (p.NC > 1) cluster_sync_all();  // partners' barriers exist before any remote access
    grid_dep_launch();
    const uint32_t tmem = tmem_base_sh;

    if (warp == 0 || warp == 6) {
        if (lane == 0) {
            if (warp == 0 && p.NC > 1 && it.rank > 0 && it.host) {
                arm_forwarded_a(p, it, full, empty, peer_empty, abort);
            } else if (warp == 6 && it.c.kcb < it.c.kc) {
                // B of a split ring (a role whose B chunks are kcb wide: its own tensor map)
                produce_b_ring(p, it, it.host ? &bmap_host : &bmap, smem, b_full, b_empty, abort);
            } else {
                produce(p, it, it.host ? &bmap_host : &bmap, smem, full, empty, abort, warp == 0, kUmmaB);
            }
        }
    } else if (warp == 7) {
        if (p.NC > 1 && it.rank == 0 && it.host) forward_a(p, it, smem, full, empty, peer_empty, abort);
    } else if (warp == 1) {
        // The whole warp runs the loop (so that loop state and descriptors stay warp-uniform);
        // one elected lane issues the MMAs and commits.
        const uint32_t idesc2 = idesc_bf16_f32(128, static_cast<uint32_t>(p.N_pad));  // a block of two
        const uint32_t idesc1 = idesc_bf16_f32(64, static_cast<uint32_t>(p.N_pad));   // one tile row
        const bool leader = elect_one();
        long long i = 0, ib = 0;
        uint64_t* last_bar = nullptr;
        uint32_t last_par = 0;
        for (int ui = 0; ui < it.count; ++ui) {
            const int ab = ui & 1;
            if (ui >= 2 && !mbar_wait(&acc_empty[ab], static_cast<uint32_t>(((ui >> 1) - 1) & 1), abort, p.st,
                                      DAK_ERR_TIMEOUT, W_MMA_ACC)) {
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + static_cast<uint32_t>(ab) * acc_stride;
            const Piece q = piece_of<PAIRS ? 1 : 0>(p, it, ui);
            const uint32_t idesc = q.m128 ? idesc2 : idesc1;
            const uint32_t kg_bytes = q.m128 ? 2048u : 1024u;  // one k-group of the block's A
            bool ok = true;
            for (int k0 = q.k0; k0 < q.k1; k0 += it.c.kc, ++i) {
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
                const int kce = min(it.c.kc, q.k1 - k0);
                const uint32_t a_base = smem_u32(smem + static_cast<size_t>(s) * it.c.stage_bytes);
                // A: no swizzle, K-major; 8x8 blocks of one k-group are 128 B apart along M,
                // k-groups are 128 (or 64) rows x 16 B = 2048 (1024) B apart along K, two per
                // MMA. B: 128-byte swizzle, K-major; 8-row groups 1024 B apart, 64-column
                // blocks N_pad x 128 B apart, +32 B per 16 columns inside a block.
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
                    const uint64_t ad0 =
                        smem_desc(a_base + static_cast<uint32_t>(k_sub >> 3) * kg_bytes, kg_bytes, 128u, 0u);
                    const uint64_t bd0 = smem_desc(b_base, 16u, 1024u, 2u);
                    if (leader) {
                        issue_mmas(d_tmem, ad0, bd0, static_cast<uint32_t>(bblk_bytes >> 4), kcs >> 4, idesc,
                                   k0 > q.k0 || k_sub > 0, (2u * kg_bytes) >> 4);
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
            last_par = static_cast<uint32_t>((ui >> 1) & 1);
        }
        if (last_bar) {  // every issued MMA has finished before TMEM is released
            volatile int dummy = 0;
            mbar_wait(last_bar, last_par, &dummy, p.st, DAK_ERR_TIMEOUT, W_DRAIN);
        }
        __syncwarp();
    } else {
        // epilogue warps 2..5 -> TMEM sub-partitions 2, 3, 0, 1 (epilogue_unit has the row map)
        const int qp = warp & 3;
        const int n_off = p.NC > 1 ? it.rank * p.N_pad : 0;  // first hidden-state row of this CTA's block
        const int e = threadIdx.x - 64;  // 0..127
        grid_dep_wait();  // C and the split workspace may still be in use by the previous kernel of the stream
        const float* rsc = nullptr;
        if (fr) {
            // r_n of the consumed normalisation: thread e sums tile rows gi, gi + G, ... of one
            // n in order (G groups), then the groups in order (host-checked N <= kFuseMaxN)
            const int G = max(1, 128 / p.N);
            if (e < G * p.N) {
                const int n = e % p.N, gi = e / p.N;
                float v = 0.f;
                for (int t = gi; t < p.ss_tiles; t += G) v += p.ss_in[static_cast<long long>(t) * p.N + n];
                fuse_red[gi * p.N + n] = v;
            }
            epilogue_bar_sync();
            if (e < p.N) {
                float v = 0.f;
                for (int gi = 0; gi < G; ++gi) v += fuse_red[gi * p.N + e];
                fuse_r[e] = rsqrtf(v * p.ss_inv_d + p.ss_eps);
            }
            epilogue_bar_sync();
            rsc = fuse_r;
        }
        bool failed = false;
        const bool xpre_on = fx && p.N_pad <= kFusePreloadN;
        float xpre[kFusePreloadN];
        float gpre = 0.f;
        for (int ui = 0; ui < it.count; ++ui) {
            const int ab = ui & 1;
            const Piece pc = piece_of<PAIRS ? 1 : 0>(p, it, ui);
            if (xpre_on) preload_x(p, pc, e, block_row_of_lane(pc.m128, qp, lane), xpre, gpre);
            if (!failed && !mbar_wait(&acc_full[ab], static_cast<uint32_t>((ui >> 1) & 1), abort, p.st,
                                      DAK_ERR_TIMEOUT, W_EPI_ACC)) {
                failed = true;
            }
            if (failed && p.P == 1 && !fx) break;  // no barrier to keep meeting
            tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(qp * 32) << 16) + static_cast<uint32_t>(ab) * acc_stride;
            epilogue_unit(p, pc, taddr, failed, &acc_empty[ab], warp, lane, e, n_off, fx, fr, rsc, fuse_ssw,
                                &last_piece, xpre_on, xpre, gpre);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (p.NC > 1) cluster_sync_all();  // no CTA leaves while a partner may still touch its shared memory
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
}

// ======================================================================================
// Chains of GEMMs in one persistent launch (N = 2..128, tensor cores). Every CTA takes its
// units of operation 0, then of operation 1, and so on, each operation dealt to its tiers'
// CTAs exactly as a launch of its own would deal it. The A producer streams the weights of
// the next operation as soon as ring slots free up, so the weight stream does not stop at
// an operation boundary (the weights never depend on an earlier operation). An operation
// marked after_prev reads its hidden states (B), and any fused-norm input, from the
// previous operation's outputs: its B loads and its epilogue wait until every CTA of the
// launch has counted the previous operation done (a device counter per operation; each
// CTA counts itself in after its last store of that operation, with release semantics,
// and only after it has itself seen the previous operation done, so the order is
// transitive). The waits are bounded like every other wait of the library.
// ======================================================================================
struct ChainParams {
    GemmParams op[kMaxChainOps];
    int after_prev[kMaxChainOps];
    int rot[kMaxChainOps];  // operation j deals its units to CTAs from rot[j] on (round the launch)
    int n_ops;
    int n_ctas;  // CTAs of the launch: every one counts itself in after every operation
    int* done;   // [n_ops] CTAs that finished operation j; the last CTA of the launch zeroes them
    DevStatus* st;
};

struct ChainMaps {
    CUtensorMap m[kMaxChainOps];  // B of each operation
};

// Units dealt by size (an independent chain all in HBM): every unit of the chain goes to
// the CTA with the least work so far, longest first, so that operations whose units differ
// in size (a 1.8 MB tile row of a K = 14336 matrix beside 0.5 MB ones) even out over the
// launch instead of landing on the same CTAs. Which CTA computes a unit does not change
// its result. n = 0: each operation deals its units round the launch from rot[j].
constexpr int kChainListMax = 4096;   // units of such a chain
constexpr int kChainListCtas = 256;   // CTAs of its launch
struct ChainList {
    int n;                                 // entries (0: not used)
    uint16_t start[kChainListCtas + 1];    // CTA c's entries are e[start[c] .. start[c + 1])
    uint16_t e[kChainListMax];             // (operation << 13) | unit, by operation then unit
};
static_assert(kMaxChainOps <= 8, "three bits of operation in a list entry");
// kernel parameters beyond 4 KB (up to 32764 bytes) need CUDA 12.1 and a Volta or later GPU
static_assert(sizeof(ChainParams) + sizeof(ChainMaps) + sizeof(ChainList) <= 32764,
              "chain parameters exceed the kernel parameter space");

enum : uint32_t { W_CHAIN_DEP = 20 };

// Wait (bounded) until *addr >= target, with acquire semantics; then order this thread's later
// asynchronous-proxy reads (bulk tensor copies) after the acquire.
__device__ __forceinline__ bool wait_count(const int* addr, int target, volatile int* abort, DevStatus* st,
                                           uint32_t where) {
    const uint64_t t0 = globaltimer();
    while (true) {
        int v;
        asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
        if (v >= target) {
            asm volatile("fence.proxy.async.global;" ::: "memory");
            return true;
        }
        if (*abort) return false;
        if (globaltimer() - t0 > kWaitLimitNs) {
            *abort = 1;
            report(st, DAK_ERR_TIMEOUT, (static_cast<unsigned long long>(where) << 32) | blockIdx.x);
            return false;
        }
        __nanosleep(128);
    }
}

// One CTA's units of operation j of a chain: the operation's own dealing (as tiles_of_cta)
// over the launch's CTAs counted from rot[j], so that operations with fewer CTAs than the
// launch do not all land on the same ones; none for a CTA beyond the operation's own CTAs.
// With a list (every unit in HBM): the CTA's entries of operation j, it.first the first
// entry's index in the list (chain_piece reads the unit from it).
__device__ __forceinline__ TileIter chain_tiles(const ChainParams& cp, const ChainList& cl, int j, int W) {
    const GemmParams& p = cp.op[j];
    if (cl.n > 0) {
        TileIter it = tiles_of_cta(p, p.n_host_ctas);  // an HBM CTA's chunking and base
        it.window = W;
        const int e0 = cl.start[blockIdx.x], e1 = cl.start[blockIdx.x + 1];
        int a = e0;
        while (a < e1 && (cl.e[a] >> 13) < j) ++a;
        int b = a;
        while (b < e1 && (cl.e[b] >> 13) == j) ++b;
        it.first = a;
        it.stride = 0;
        it.count = b - a;
        return it;
    }
    const int cta = (static_cast<int>(blockIdx.x) + cp.n_ctas - cp.rot[j]) % cp.n_ctas;
    TileIter it = tiles_of_cta(p, cta);
    it.window = W;
    if (cta >= p.n_host_ctas + p.n_hbm_ctas) it.count = 0;
    return it;
}

// The ui-th unit of chain_tiles' iteration
__device__ __forceinline__ Piece chain_piece(const ChainList& cl, const GemmParams& p, TileIter it, int ui) {
    if (cl.n > 0) {
        it.first = cl.e[it.first + ui] & 0x1fff;
        return piece_of(p, it, 0);
    }
    return piece_of(p, it, ui);
}

// A or B producer of a chain: the chunks of every operation in order, ring index i running
// on across operations. The B producer waits for an operation's inputs before its first copy.
__device__ __forceinline__ void chain_produce(const ChainParams& cp, const ChainMaps& maps, const ChainList& cl,
                                              uint8_t* smem,
                                              uint64_t* full, uint64_t* empty, volatile int* abort, bool is_a,
                                              int W) {
    const uint64_t pol_a = policy_evict_first();
    long long i = 0;
    for (int j = 0; j < cp.n_ops && !*abort; ++j) {
        const GemmParams& p = cp.op[j];
        const TileIter it = chain_tiles(cp, cl, j, W);
        if (!is_a) {
            if (j == 0) {
                grid_dep_wait();  // the first operation's hidden states may come from the previous kernel
            } else if (cp.after_prev[j] && !wait_count(cp.done + (j - 1), cp.n_ctas, abort, cp.st, W_CHAIN_DEP)) {
                break;
            }
        }
        for (int ui = 0; ui < it.count && !*abort; ++ui) {
            const Piece q = chain_piece(cl, p, it, ui);
            const uint8_t* src = block_src(p, it, q);
            const int cb = col_bytes(q);
            for (int k0 = q.k0; k0 < q.k1; k0 += it.c.kc, ++i) {
                const int s = static_cast<int>(i % W);
                if (i >= W && !mbar_wait(&empty[s], static_cast<uint32_t>(((i / W) - 1) & 1), abort, p.st,
                                         DAK_ERR_TIMEOUT, is_a ? W_PROD_EMPTY : W_BPROD_EMPTY)) {
                    goto done;
                }
                uint8_t* dst = smem + static_cast<size_t>(s) * it.c.stage_bytes;
                if (is_a) {
                    const uint32_t a_bytes = static_cast<uint32_t>(min(it.c.kc, q.k1 - k0) * cb);
                    mbar_arrive_expect_tx(&full[s], a_bytes);
                    bulk_g2s(dst, src + static_cast<long long>(k0) * cb, a_bytes, &full[s], pol_a);
                } else {
                    mbar_arrive_expect_tx(&full[s], b_stage_bytes(p, kUmmaB, it.c.kcb));
                    issue_b(p, &maps.m[j], dst + it.c.kc * it.c.a_cb, k0, &full[s], kUmmaB, 0, it.c.kcb);
                }
            }
        }
    }
done:
    drain_fills(full, W, i, cp.st);
}

template <bool F>
__global__ void __launch_bounds__(kUmmaThreads, 1)
    gemm_chain_kernel(const __grid_constant__ ChainParams cp, const __grid_constant__ ChainMaps maps,
                      const __grid_constant__ ChainList cl) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint64_t full[8], empty[8], acc_full[2], acc_empty[2];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;
    __shared__ int last_piece;
    __shared__ float fuse_ssw[4][kFuseMaxN];
    __shared__ float fuse_red[kFuseMaxN];
    __shared__ float fuse_r[kFuseMaxN];
    volatile int* abort = &abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N_pad = cp.op[0].N_pad;      // the same for every operation of a chain
    const int W = cp.op[0].ch[0].stages;  // one ring for every operation and tier
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint32_t tmem_cols = 32;
    while (tmem_cols < static_cast<uint32_t>(2 * N_pad)) tmem_cols <<= 1;
    const uint32_t acc_stride = tmem_cols >> 1;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < W; ++s) {
            mbar_init(&full[s], 2);   // A producer + B producer
            mbar_init(&empty[s], 1);  // MMA commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        fence_mbar_init();
        for (int j = 0; j < cp.n_ops; ++j) prefetch_tmap(&maps.m[j]);
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base_sh, tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    grid_dep_launch();
    const uint32_t tmem = tmem_base_sh;

    if (warp == 0 || warp == 6) {
        if (lane == 0) chain_produce(cp, maps, cl, smem, full, empty, abort, warp == 0, W);
    } else if (warp == 1) {
        const uint32_t idesc2 = idesc_bf16_f32(128, static_cast<uint32_t>(N_pad));  // a block of two
        const uint32_t idesc1 = idesc_bf16_f32(64, static_cast<uint32_t>(N_pad));   // one tile row
        const bool leader = elect_one();
        const int a_stage_bytes = cp.op[0].ch[0].kc * cp.op[0].ch[0].a_cb;
        const uint32_t bblk16 = static_cast<uint32_t>((N_pad * 128) >> 4);
        long long i = 0;
        int uu = 0;  // units of the whole chain so far (the accumulator alternates on it)
        uint64_t* last_bar = nullptr;
        uint32_t last_par = 0;
        bool ok = true;
        for (int j = 0; j < cp.n_ops && ok; ++j) {
            const GemmParams& p = cp.op[j];
            const TileIter it = chain_tiles(cp, cl, j, W);
            for (int ui = 0; ui < it.count && ok; ++ui, ++uu) {
                const int ab = uu & 1;
                if (uu >= 2 && !mbar_wait(&acc_empty[ab], static_cast<uint32_t>(((uu >> 1) - 1) & 1), abort, p.st,
                                          DAK_ERR_TIMEOUT, W_MMA_ACC)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + static_cast<uint32_t>(ab) * acc_stride;
                const Piece q = chain_piece(cl, p, it, ui);
                const uint32_t idesc = q.m128 ? idesc2 : idesc1;
                const uint32_t kg_bytes = q.m128 ? 2048u : 1024u;
                for (int k0 = q.k0; k0 < q.k1; k0 += it.c.kc, ++i) {
                    const int s = static_cast<int>(i % W);
                    if (!mbar_wait(&full[s], static_cast<uint32_t>((i / W) & 1), abort, p.st, DAK_ERR_TIMEOUT,
                                   W_MMA_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int kce = min(it.c.kc, q.k1 - k0);
                    const uint32_t a_base = smem_u32(smem + static_cast<size_t>(s) * it.c.stage_bytes);
                    const uint64_t ad0 = smem_desc(a_base, kg_bytes, 128u, 0u);
                    const uint64_t bd0 = smem_desc(a_base + static_cast<uint32_t>(a_stage_bytes), 16u, 1024u, 2u);
                    if (leader) {
                        issue_mmas(d_tmem, ad0, bd0, bblk16, kce >> 4, idesc, k0 > q.k0, (2u * kg_bytes) >> 4);
                        umma_commit(&empty[s]);
                    }
                    __syncwarp();
                    last_bar = &empty[s];
                    last_par = static_cast<uint32_t>((i / W) & 1);
                }
                if (!ok) break;
                if (leader) umma_commit(&acc_full[ab]);
                __syncwarp();
                last_bar = &acc_full[ab];
                last_par = static_cast<uint32_t>((uu >> 1) & 1);
            }
        }
        if (last_bar) {  // every issued MMA has finished before TMEM is released
            volatile int dummy = 0;
            mbar_wait(last_bar, last_par, &dummy, cp.st, DAK_ERR_TIMEOUT, W_DRAIN);
        }
        __syncwarp();
    } else if (warp >= 2 && warp <= 5) {
        // epilogue warps 2..5 -> TMEM sub-partitions 2, 3, 0, 1 (as gemm_umma_kernel)
        const int qp = warp & 3;
        const int e = threadIdx.x - 64;  // 0..127
        grid_dep_wait();  // C, the fused inputs and the workspace may be in use by the previous kernel
        bool failed = false;
        int uu = 0;
        for (int j = 0; j < cp.n_ops; ++j) {
            const GemmParams& p = cp.op[j];
            const bool fx = F && p.res_x != nullptr;
            const bool fr = F && p.ss_in != nullptr;
            const TileIter it = chain_tiles(cp, cl, j, W);
            if (j > 0 && cp.after_prev[j]) {
                // the previous operation's outputs (this one's B, fused inputs, or a buffer it
                // overwrites) are complete once every CTA has counted it in
                if (e == 0 && !failed && !wait_count(cp.done + (j - 1), cp.n_ctas, abort, cp.st, W_CHAIN_DEP))
                    failed = true;
                epilogue_bar_sync();
                failed = failed || *abort;
            }
            const float* rsc = nullptr;
            if (fr) {
                const int G = max(1, 128 / p.N);
                if (e < G * p.N) {
                    const int n = e % p.N, gi = e / p.N;
                    float v = 0.f;
                    for (int t = gi; t < p.ss_tiles; t += G) v += p.ss_in[static_cast<long long>(t) * p.N + n];
                    fuse_red[gi * p.N + n] = v;
                }
                epilogue_bar_sync();
                if (e < p.N) {
                    float v = 0.f;
                    for (int gi = 0; gi < G; ++gi) v += fuse_red[gi * p.N + e];
                    fuse_r[e] = rsqrtf(v * p.ss_inv_d + p.ss_eps);
                }
                epilogue_bar_sync();
                rsc = fuse_r;
            }
            const bool xpre_on = fx && N_pad <= kFusePreloadN;
            float xpre[kFusePreloadN];
            float gpre = 0.f;
            for (int ui = 0; ui < it.count; ++ui, ++uu) {
                const int ab = uu & 1;
                const Piece pc = chain_piece(cl, p, it, ui);
                if (xpre_on) preload_x(p, pc, e, block_row_of_lane(pc.m128, qp, lane), xpre, gpre);
                if (!failed && !mbar_wait(&acc_full[ab], static_cast<uint32_t>((uu >> 1) & 1), abort, p.st,
                                          DAK_ERR_TIMEOUT, W_EPI_ACC)) {
                    failed = true;
                }
                tc_fence_after();
                const uint32_t taddr =
                    tmem + (static_cast<uint32_t>(qp * 32) << 16) + static_cast<uint32_t>(ab) * acc_stride;
                epilogue_unit(p, pc, taddr, failed, &acc_empty[ab], warp, lane, e, 0, fx, fr, rsc, fuse_ssw,
                              &last_piece, xpre_on, xpre, gpre);
            }
            // this CTA is done with operation j: every epilogue thread's stores are ordered
            // before the count by the barrier, and made visible at GPU scope (and to the
            // bulk copies that read them) before it
            epilogue_bar_sync();
            if (e == 0 && !failed && !*abort) {
                asm volatile("fence.proxy.async.global;" ::: "memory");
                __threadfence();
                const int before = atomic_add_acq_rel(cp.done + j, 1);
                if (j == cp.n_ops - 1 && before == cp.n_ctas - 1) {
                    // every CTA has finished every operation: ready for the next launch
                    for (int jj = 0; jj < cp.n_ops; ++jj) cp.done[jj] = 0;
                    __threadfence();
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
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
    if (!enc || fault_due(DAK_FAULT_TENSOR_MAP)) return false;
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
// Default cap on CTAs reading host tiles (the congestion cap of section 4.3.1). One CTA per
// tile row: 48, measured best for the decode step (more host bytes in flight at once). Wide
// B (clusters sharing tile rows): 32 CTAs, i.e. 32 / NC clusters, since there the HBM side
// needs its SMs for the N_pad = 256 tensor work.
constexpr int kDefaultHostCtas = 48;
constexpr int kDefaultHostCtasWide = 32;
constexpr int kMaxBlockN = 256;          // hidden-state rows of one CTA's tile
constexpr int kMaxWideN = 4 * kMaxBlockN;  // rows of one launch: a cluster of up to 4 CTAs shares A
constexpr int kDefaultHostWindow = 4;

// Launch with the optional cluster dimension and programmatic-dependent-launch attribute.
template <typename Kernel, typename... Args>
static cudaError_t launch_ex(Kernel k, int grid, int threads, int smem, int cluster, bool pdl, cudaStream_t s,
                             const Args&... args) {
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
    return cudaLaunchKernelEx(&cfg, k, args...);
}

// Clusters of `cluster` CTAs of kernel k (threads, smem) that the device holds at once: a
// cluster's CTAs share a GPC, so clusters of 4 leave the SMs of a GPC beyond a multiple of 4
// idle and fewer than sms / 4 fit. A persistent grid sized for more clusters than fit runs
// the extra ones after the others, a whole tail. Cached per device and shape; 0 when the
// query fails (the caller then assumes sms / cluster).
template <typename Kernel>
static int max_active_clusters(Kernel k, int threads, int smem, int cluster) {
    struct Key {
        int dev, threads, smem, cluster;
        const void* fn;
    };
    static std::mutex mu;
    static std::vector<std::pair<Key, int>> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const Key key{dev, threads, smem, cluster, reinterpret_cast<const void*>(k)};
    std::lock_guard<std::mutex> lock(mu);
    for (const auto& e : cache) {
        const Key& c = e.first;
        if (c.dev == key.dev && c.threads == key.threads && c.smem == key.smem && c.cluster == key.cluster &&
            c.fn == key.fn)
            return e.second;
    }
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(cluster * 64));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    cache.push_back({key, n});
    return n;
}

// Workspace of split tile rows: fp32 partial tiles and one counter per tile row, in device
// memory that the module owns (no allocation at launch time, so launches can be captured in
// CUDA graphs). Launches on one stream use it in turn (the partials and counters are touched
// only after the previous kernel of the stream has finished); launches that split tile rows
// must not run concurrently on different streams of one device.
constexpr long long kSplitFloats = 8ll << 20;  // 32 MiB
constexpr int kSplitTiles = 1 << 16;
static __device__ float g_split_part[kSplitFloats];
static __device__ int g_split_cnt[kSplitTiles];

// The arrays' device addresses on the current device, looked up once per device and context
// (after cudaDeviceReset they live at new addresses of a new context).
static bool split_workspace(float** part, int** cnt) {
    static float* parts[64];
    static int* cnts[64];
    static unsigned long long ctx[64];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long id = current_context_id();
    if (!parts[dev] || !cnts[dev] || ctx[dev] != id) {
        void* a = nullptr;
        void* b = nullptr;
        if (cudaGetSymbolAddress(&a, g_split_part) != cudaSuccess || cudaGetSymbolAddress(&b, g_split_cnt) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        parts[dev] = static_cast<float*>(a);
        cnts[dev] = static_cast<int*>(b);
        ctx[dev] = current_context_id();
    }
    *part = parts[dev];
    *cnt = cnts[dev];
    return true;
}

// Pieces per block: the split of each block's K range into P parts (at multiples of 64
// columns), chosen from the shape and the SM count only, never from the placement, so that
// results are bit-identical across offload ratios. Automatic, in two steps:
//  1. the all-HBM cost of each P in 1..8: the busiest CTA's time, ceil(B P / slots) waves of
//     (1 / P of a block's bytes plus the fixed cost of a piece), B = T blocks of one tile row
//     or ceil(T / 2) pair blocks (rows = 2). The fixed cost, piece_us of a CTA streaming at
//     about 62 GB/s, is fitted to decode steps on this GPU: on the tensor cores
//     max(1, N_pad / 16) us (the partial tile of 64 x N_pad fp32, the count, the last
//     piece's sum, a ragged last chunk), on the CUDA cores 2 us (there the consumers that
//     run the FMAs also store the partial rows). An unsplit block pays half of it (its
//     epilogue stores C only).
//  2. among the P within 3% of the lowest cost, the smallest whose pieces give a host part
//     of a tenth of the blocks at least as many units as the host CTA cap (a small host
//     part spread over more CTAs keeps more host bytes in flight), else the cheapest.
// Pieces keep at least 512 columns and the workspace must hold the partials (T tile rows'
// worth; the bound used, T + 2, leaves room to spare).
// tuning.split_k > 0 fixes P (1 = no split).
constexpr double kCtaStreamBytesPerUs = 62.5e3;
// bf16 tensor rate of one SM issuing M = 64 tiles, FLOP per us (fitted: the 8B gate+up at 256
// rows, 448 tile rows in three waves on 150 SMs, took 104 us all-HBM), and the host link's
// read rate, bytes per us (the read-stream probe: 211 GB/s)
constexpr double kSmTensorFlopsPerUs = 3.76e6;
constexpr double kHostLinkBytesPerUs = 2.1e5;
constexpr double kHostCtaBytesPerUs = 1.3e4;  // a host CTA through tensor-bound tile rows (fitted: 512 KiB in ~40 us)
// The same two rates for 128-row tiles (M = 128 MMAs), fitted to the 8B gate+up at N = 1024
// in 128-row tiles: 224 tiles in 7 waves of 32 clusters took 234 us all-HBM (33 us per
// M = 128 x N = 256 x K = 4096 unit), and at x = 0.25 a host cluster took ~96 us per 1 MiB
// tile while the link was not yet full.
constexpr double kSmTensorFlopsPerUs128 = 8.1e6;
constexpr double kHostCtaBytesPerUs128 = 1.09e4;

static int split_pieces(int T, int K_pad, int N_pad, int slots, long long tile_bytes, int host_cap, int pstep,
                        double piece_us, long long max_tiles, long long max_floats, const dak_tuning* t, int rows) {
    const int steps = (K_pad + 63) / 64;
    auto fits = [&](int P) {
        return P <= (K_pad + pstep - 1) / pstep && T <= max_tiles &&
               static_cast<long long>(T + 2) * P * kTileM * N_pad <= max_floats;
    };
    if (t && t->split_k > 0) {
        int P = std::min(kMaxPieces, t->split_k);
        while (P > 1 && !fits(P)) --P;
        return P;
    }
    const double c = piece_us * kCtaStreamBytesPerUs / (static_cast<double>(rows) * tile_bytes);  // in blocks
    const long long nb = blocks_of(T, rows == 2);
    double cost[kMaxPieces + 1] = {};
    int top = 1;
    for (int P = 1; P <= kMaxPieces; ++P) {
        if (P > 1 && (!fits(P) || steps / P < kMinPieceSteps)) break;
        const long long waves = (nb * P + slots - 1) / slots;
        cost[P] = static_cast<double>(waves) * (1.0 / P + (P > 1 ? c : 0.5 * c));
        top = P;
    }
    int cheapest = 1;
    for (int P = 2; P <= top; ++P)
        if (cost[P] < cost[cheapest]) cheapest = P;
    const int h_small = blocks_of((T + 9) / 10, rows == 2);
    for (int P = 1; P <= top; ++P)
        if (cost[P] <= 1.03 * cost[cheapest] && h_small * P >= host_cap) return P;
    return cheapest;
}

// A caller's workspace: the per-tile-row counters of every launch that uses it (a fixed
// region, indexed by tile row, so that launches over different matrices can share it), then
// the partial tiles.
constexpr long long kCallerCounterBytes = static_cast<long long>(kSplitTiles) * 4;

size_t gemm_workspace_bytes(const dak_placement* A, int N) {
    if (!A || A->kind != 0 || N < 1) return 0;
    if (N > kMaxBlockN || A->T > kSplitTiles) return 0;  // never split
    const long long n_pad = (N + 15) & ~15;
    return static_cast<size_t>(kCallerCounterBytes +
                               static_cast<long long>(A->T + 2) * kMaxPieces * kTileM * n_pad * 4);
}

void reset_split_counters() {
    float* part = nullptr;
    int* cnt = nullptr;
    if (split_workspace(&part, &cnt)) cudaMemset(cnt, 0, sizeof(int) * kSplitTiles);
}

// Everything one launch decides from the shape, the SM count and the tuning: the rings'
// layout, the pieces per tile row and the CTAs of each role. Host arithmetic only (no CUDA
// call), so that dak_gemm_plan can report it without a GPU.
struct BlockPlan {
    bool umma;
    int pairs;  // 128-row tiles: pair blocks (M = 128)
    int cl_slots;  // clusters (of NC CTAs) the schedule assumes the device holds at once
    int NC, N_pad, P, pstep, kcb, kcb_host, smem, grid;  // kcb / kcb_host: B chunk width of each role's map
    Chunks ch[2];  // [0] HBM-side CTAs, [1] host-side CTAs
    int n_host_ctas, n_hbm_ctas, host_window, hbm_window;
};

// T tile rows of 64 (h of them on the host) of K_pad columns, tile_bytes each; N
// hidden-state rows (at most one launch's worth); caller_ws: the partial tiles go to a
// caller's workspace of ws_bytes; pairs: a placement of 128-row tiles (T and h even), whose
// blocks of two tile rows are the units of work.
// tensor_cores: plan the tcgen05 kernel at N = 1 too (a chain has no CUDA-core path)
static dak_status plan_block(int T, int h, int K_pad, long long tile_bytes, int N, int sms, const dak_tuning* t,
                             bool caller_ws, size_t ws_bytes, BlockPlan* bp, int pairs, int cluster_slots = 0,
                             bool tensor_cores = false) {
    if (N < 1 || N > kMaxWideN || sms < 1) return DAK_ERR_INVALID;
    BlockPlan& q = *bp;
    q = BlockPlan{};
    // wide B: NC CTAs of a cluster share each tile row, CTA r computing rows [256 r, 256 r + 256)
    q.NC = N > kMaxBlockN ? (N + kMaxBlockN - 1) / kMaxBlockN : 1;
    q.P = 1;
    q.umma = N >= 2 || tensor_cores;  // N = 2..7 padded to 8 columns: measured 1.2-2.7x faster than FMA
    q.pstep = q.umma ? 64 : 256;      // the B block of the tensor-core / CUDA-core layout
    const bool umma = q.umma;
    if (pairs && ((T | h) & 1)) return DAK_ERR_INVALID;
    q.pairs = pairs ? 1 : 0;
    // (pair blocks on the tensor cores: a multiple of 16, the N step of M = 128 MMAs)
    q.N_pad = N > kMaxBlockN ? kMaxBlockN : ((q.pairs && umma) ? (N + 15) & ~15 : (N + 7) & ~7);
    const int rows_b = umma ? q.N_pad : N;
    const int NC = q.NC;
    const int cb_hbm = q.pairs ? 256 : 128;  // bytes of A per column in a stage (both roles)
    // a stage: A (k x cb bytes: one tile row, or two), then B (k x 2 bytes per hidden-state row)
    auto stage_cb = [&](int k, int cb) { return (k * cb + k * 2 * rows_b + 1023) & ~1023; };
    auto stage_of = [&](int k) { return stage_cb(k, cb_hbm); };

    int per_sm = 1;
    if (umma && NC == 1 && t && (t->ctas_per_sm == 1 || t->ctas_per_sm == 2)) per_sm = t->ctas_per_sm;
    const int budget = per_sm == 2 ? kSmemBudgetTwoPerSm : kSmemBudget;
    int kc;
    if (t && t->chunk_k > 0) {
        kc = t->chunk_k;
    } else if (!umma) {
        kc = q.pairs ? 256 : 512;  // 64 KiB of A per stage
    } else if (per_sm == 2) {
        // the widest chunk that leaves two stages
        kc = 64;
        for (int cand : {512, 384, 256, 192, 128}) {
            if (2 * stage_of(cand) + 1024 <= budget) {
                kc = cand;
                break;
            }
        }
    } else {
        // the widest chunk (up to 512 columns, 64 KiB of A) of which two stages fit: per-chunk
        // costs dominate a CTA's stream, so two wide stages beat three narrow ones (measured
        // at x = 0: N = 64 at 384 columns 15% faster than at 256, N = 128 at 256 columns 25%
        // faster than at 128, N = 256 at 128 columns 30% faster than at 64)
        kc = 64;
        for (int cand : {512, 448, 384, 320, 256, 192, 128}) {
            if (2 * stage_of(cand) + 1024 <= budget) {
                kc = cand;
                break;
            }
        }
    }
    if (kc % 64 != 0 || kc > 1024 || (!umma && kc % 256 != 0)) return DAK_ERR_INVALID;
    // Ring layouts. Shared tile rows (NC > 1): A in 256-column chunks and B through its own
    // ring of 64-column chunks, so that A copies and forwards stay large while B fills the
    // rest. One CTA per tile row: the unified ring for both tiers, except that with wide B
    // (N_pad > 128, where two unified stages hold only 128 columns of A) CTAs reading host
    // tiles take the split layout: 32 KiB A chunks in three or four stages keep about three
    // times the host bytes in flight, and host reads are latency-bound (a tensor-bound
    // linear at N = 256 ran its host tile rows 1.3x slower than its HBM ones without it).
    // That role's B chunks are 64 columns wide, so it gets a tensor map of its own.
    // Clusters (NC > 1): host tile rows are forwarded by rank 0 (A-only slots, split layout);
    // HBM tile rows are streamed by every rank and take the unified ring like N_pad = 256 alone.
    const bool b_ring_all = false;
    const bool b_ring_host = umma && (NC > 1 || (q.N_pad > 128 && kc <= 128 && !(t && t->chunk_k > 0)));
    // (NC > 1: each CTA holds 2 x 256 TMEM columns, the whole TMEM of an SM: one CTA per SM)
    const int CL = NC;  // CTAs per cluster
    auto layout = [&](int kc_, bool split, int cb, Chunks* L) -> bool {
        L->kc = kc_;
        L->kcb = split ? 64 : kc_;
        L->a_cb = cb;
        if (split) {
            L->stage_bytes = (kc_ * cb + 1023) & ~1023;
            L->b_slot_bytes = (q.N_pad * L->kcb * 2 + 1023) & ~1023;
            const int avail = budget - 1024;
            L->stages = std::min(4, std::max(2, avail / 2 / L->stage_bytes));  // about half for A
            L->wb = std::min(8, (avail - L->stages * L->stage_bytes) / L->b_slot_bytes);
            if (L->wb < 2) {
                L->stages = 2;
                L->wb = std::min(8, (avail - L->stages * L->stage_bytes) / L->b_slot_bytes);
            }
            if (L->wb < 2) return false;
        } else {
            L->stage_bytes = stage_cb(kc_, cb);
            L->stages = std::min(8, (budget - (umma ? 1024 : 0)) / L->stage_bytes);
            L->wb = 0;
            L->b_slot_bytes = 0;
            if (L->stages < 1 || (L->stages < 2 && !(t && t->chunk_k > 0))) return false;
        }
        L->b_ring_off = L->stages * L->stage_bytes;
        return true;
    };
    if (!layout(kc, b_ring_all, cb_hbm, &q.ch[0])) return DAK_ERR_INVALID;
    q.ch[1] = q.ch[0];
    if (!b_ring_all && b_ring_host && h > 0) {
        // 32 KiB of A per chunk
        const int kch = (NC > 1 && t && t->chunk_k > 0) ? std::max(64, t->chunk_k) : (q.pairs ? 128 : 256);
        Chunks L;
        if (layout(kch, true, cb_hbm, &L)) {
            q.ch[1] = L;
        } else if (NC > 1) {
            return DAK_ERR_INVALID;  // a forwarding cluster needs A-only slots
        }
    }
    q.kcb = q.ch[0].kcb;
    q.kcb_host = q.ch[1].kcb;
    auto ring_bytes = [](const Chunks& L) { return L.stages * L.stage_bytes + L.wb * L.b_slot_bytes; };
    const int rings = std::max(ring_bytes(q.ch[0]), ring_bytes(q.ch[1]));
    q.smem = rings + (umma ? 1024 : 0);
    const int max_stages = std::max(q.ch[0].stages, q.ch[1].stages);
    const int hb = blocks_of(h, q.pairs), gb = blocks_of(T - h, q.pairs);  // blocks: units before the split

    // pieces per block (one CTA per block's columns; automatic only while the tile rows are
    // memory-bound, N_pad <= 128: at N_pad = 256 the tensor work of a tile row is what the
    // split would spread, and the partial tiles cost more than it saves)
    if (NC == 1 && (q.N_pad <= 128 || (t && t->split_k > 0))) {
        const double piece_us = umma ? std::max(1.0, q.N_pad / 16.0) : 2.0;
        // the caller's workspace (counters, then partial tiles) or the module's own
        const long long cnt_bytes = caller_ws ? kCallerCounterBytes : 0;
        const long long max_floats =
            caller_ws ? std::max(0ll, (static_cast<long long>(ws_bytes) - cnt_bytes) / 4) : kSplitFloats;
        q.P = split_pieces(T, K_pad, q.N_pad, sms * per_sm, tile_bytes, kDefaultHostCtas, q.pstep, piece_us,
                           kSplitTiles, max_floats, t, q.pairs ? 2 : 1);
    }

    // schedule in cluster units; a role's units are its tile rows x P pieces; cluster_slots
    // (when known): the clusters the device holds at once
    const int cs = (t && t->cluster_slots > 0) ? t->cluster_slots : cluster_slots;
    const int cl_slots = std::max(1, (CL > 1 && cs > 0) ? std::min(cs, (sms * per_sm) / CL) : (sms * per_sm) / CL);
    q.cl_slots = cl_slots;
    dak_tuning tc{};
    if (t) tc = *t;
    const int host_cap = NC > 1 ? kDefaultHostCtasWide : kDefaultHostCtas;
    int hc = tc.host_ctas > 0 ? tc.host_ctas : host_cap;
    if (!(tc.host_ctas > 0) && CL == 1 && hb * q.P > hc && 3 * hb * q.P <= 4 * hc) {
        hc = hb * q.P;  // up to a third over the cap: one wave of host units rather than two
    }
    // A tile row at N_pad >= 256 is tensor work: its MMAs take longer than its bytes, and
    // every host CTA is an SM taken from the HBM side's compute. There the host CTA count is
    // chosen by the time model of section 4.1 (factor 3: the two roles' times balanced, each
    // in whole waves): host time = max(waves x per-unit time of a host CTA, host bytes / link
    // rate), HBM time = waves x per-unit compute time; the count minimising the larger is
    // taken, or the largest count within 1% of it (more host CTAs keep the link busier), at
    // most the congestion cap. A host CTA of such a GEMM gets through a tile row more slowly
    // than an HBM one (about 40 us per 512 KiB against 36 us of MMAs, measured at 256 rows),
    // so the flat segment of Fig. 6 ends before x = B_host T_comp / C. Memory-bound tile rows
    // keep the fixed cap above.
    if (q.N_pad >= 256 && h > 0 && !(t && t->host_ctas > 0)) {
        // a unit is a block's piece: one 64-row tile row (M = 64 MMAs) or a 128-row tile
        // (M = 128 MMAs, about twice the rate per SM)
        const double unit_bytes = (q.pairs ? 2.0 : 1.0) * static_cast<double>(tile_bytes) / q.P;
        const double t_mma = (q.pairs ? 2.0 : 1.0) * 2.0 * kTileM * q.N_pad * (static_cast<double>(K_pad) / q.P) /
                             (q.pairs ? kSmTensorFlopsPerUs128 : kSmTensorFlopsPerUs);
        const double t_unit = std::max(t_mma, unit_bytes / kCtaStreamBytesPerUs);
        const double t_host_unit = std::max(t_unit, unit_bytes / (q.pairs ? kHostCtaBytesPerUs128 : kHostCtaBytesPerUs));
        const double t_link = static_cast<double>(h) * tile_bytes / kHostLinkBytesPerUs;
        const int slots = cl_slots;
        const long long hu = static_cast<long long>(hb) * q.P, gu = static_cast<long long>(gb) * q.P;
        // one SM of a host cluster reads the link (rank 0 forwards): the cap counts reading SMs
        const int n_max = static_cast<int>(std::min<long long>(std::min<long long>(hu, kDefaultHostCtas),
                                                               slots - (gu > 0 ? 1 : 0)));
        auto model = [&](int n) {  // n counts cluster units, as schedule() does
            const double th = std::max(static_cast<double>((hu + n - 1) / n) * t_host_unit, t_link);
            const int m = slots - n;
            const double tg = gu > 0 ? static_cast<double>((gu + m - 1) / m) * t_unit : 0.0;
            return std::max(th, tg);
        };
        double best = 1e300;
        for (int n = 1; n <= n_max; ++n) best = std::min(best, model(n));
        int best_n = 1;
        for (int n = 1; n <= n_max; ++n)
            if (model(n) <= 1.01 * best) best_n = n;
        hc = best_n * CL;
    }
    tc.host_ctas = std::max(1, hc / CL);
    if (tc.hbm_ctas > 0) tc.hbm_ctas = std::max(1, tc.hbm_ctas / CL);
    const Sched sc = schedule(hb * q.P, gb * q.P, cl_slots, &tc,
                              std::max(1, host_cap / CL), std::min(kDefaultHostWindow, q.ch[1].stages),
                              q.ch[0].stages, max_stages);
    q.n_host_ctas = sc.n_host_ctas;
    q.n_hbm_ctas = sc.n_hbm_ctas;
    q.host_window = std::min(sc.host_window, q.ch[1].stages);
    q.hbm_window = std::min(sc.hbm_window, q.ch[0].stages);
    q.grid = (q.n_host_ctas + q.n_hbm_ctas) * CL;
    return DAK_OK;
}

// The plan of one launch over placement A on the current device: plan_block, with the
// persistent grid of a cluster launch sized to the clusters that fit at once (unless the
// tuning fixes cluster_slots).
static dak_status plan_launch(const dak_placement* A, int N, const dak_tuning* t, bool caller_ws, size_t ws_bytes,
                              BlockPlan* bp) {
    const int sms = device_sm_count();
    const int pairs = A->tile_m == 2 * kTileM;
    dak_status r = plan_block(A->T, A->h, static_cast<int>(A->K_pad), A->tile_bytes, N, sms, t, caller_ws, ws_bytes,
                              bp, pairs);
    if (r != DAK_OK || bp->NC == 1 || (t && t->cluster_slots > 0)) return r;
    const int fit = max_active_clusters(pairs ? gemm_umma_kernel<false, true> : gemm_umma_kernel<false, false>,
                                        kUmmaThreads, bp->smem, bp->NC);
    if (fit > 0 && fit < sms / bp->NC)
        r = plan_block(A->T, A->h, static_cast<int>(A->K_pad), A->tile_bytes, N, sms, t, caller_ws, ws_bytes, bp,
                       pairs, fit);
    return r;
}

// One launch over up to kMaxWideN hidden-state rows: one CTA per tile row up to 256 rows
// (the widest tcgen05 tile used here), a cluster of ceil(N / 256) CTAs per tile row beyond.
static dak_status launch_gemm_block(const dak_placement* A, const void* host_src, const void* B, void* C, int N,
                                    int c_fp32, const dak_tuning* t, void* ws, size_t ws_bytes, cudaStream_t stream,
                                    const GemmFuse* fuse, const LinkHandoff* link) {
    if (!A || A->kind != 0) return DAK_ERR_INVALID;
    if (N < 1 || N > kMaxWideN) return DAK_ERR_INVALID;
    if (A->M == 0 || A->T == 0) return DAK_OK;  // nothing to compute; C may be empty
    if (!B || !C) return DAK_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(B) & 15) || (reinterpret_cast<uintptr_t>(C) & 15)) return DAK_ERR_ALIGN;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DAK_ERR_CUDA;
    if (dev != A->device) return DAK_ERR_INVALID;

    BlockPlan bp;
    const dak_status r = plan_launch(A, N, t, ws != nullptr, ws_bytes, &bp);
    if (r != DAK_OK) return r;
    if (bp.grid == 0) return DAK_OK;

    GemmParams p{};
    p.a_host = static_cast<const uint8_t*>(host_src);
    p.a_hbm = static_cast<const uint8_t*>(A->hbm_ptr);
    p.B = static_cast<const __nv_bfloat16*>(B);
    p.C = C;
    p.M = static_cast<int>(A->M);
    p.K = static_cast<int>(A->K);
    p.K_pad = static_cast<int>(A->K_pad);
    p.N = N;
    p.NC = bp.NC;
    p.N_pad = bp.N_pad;
    p.T = A->T;
    p.h = A->h;
    p.pairs = bp.pairs;
    p.hb = blocks_of(p.h, p.pairs);
    p.gb = blocks_of(p.T - p.h, p.pairs);
    p.c_fp32 = c_fp32 ? 1 : 0;
    p.tile_bytes = A->tile_bytes;
    p.glu = A->glu;
    p.P = bp.P;
    p.pstep = bp.pstep;
    p.ch[0] = bp.ch[0];
    p.ch[1] = bp.ch[1];
    p.n_host_ctas = bp.n_host_ctas;
    p.n_hbm_ctas = bp.n_hbm_ctas;
    p.host_window = bp.host_window;
    p.hbm_window = bp.hbm_window;
    p.st = status_ptr();
    if (!p.st) return DAK_ERR_CUDA;
    if (p.h > 0 && !p.a_host) return DAK_ERR_INVALID;
    if (link && link->ctr) {
        // one signal per host cluster: its rank 0 runs the A producer (the others are fed)
        p.link = link->ctr;
        p.link_after = link->after;
    }
    if (fuse && (fuse->res_x || fuse->ss_in)) {
        if (N > kFuseMaxN || bp.NC != 1) return DAK_ERR_UNSUPPORTED;
        if (fuse->res_x) {
            if (p.glu || c_fp32 || !fuse->res_g || !fuse->ss_out) return DAK_ERR_INVALID;
            p.res_x = fuse->res_x;
            p.res_g = static_cast<const __nv_bfloat16*>(fuse->res_g);
            p.ss_out = fuse->ss_out;
        }
        if (fuse->ss_in) {
            if (fuse->ss_tiles < 1) return DAK_ERR_INVALID;
            p.ss_in = fuse->ss_in;
            p.ss_tiles = fuse->ss_tiles;
            p.ss_inv_d = fuse->inv_d;
            p.ss_eps = fuse->eps;
        }
    }
    if (p.P > 1) {
        if (ws) {
            p.cnt = static_cast<int*>(ws);
            p.part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kCallerCounterBytes);
        } else if (!split_workspace(&p.part, &p.cnt)) {
            return DAK_ERR_CUDA;
        }
    }

    alignas(64) CUtensorMap bmap, bmap_host;
    int b3d = 0, b3d_host = 0;
    if (!make_b_map(&bmap, B, p.K, N, p.N_pad, bp.kcb, bp.umma ? kUmmaB : kCoreB, &b3d)) return DAK_ERR_CUDA;
    if (bp.kcb_host != bp.kcb) {
        if (!make_b_map(&bmap_host, B, p.K, N, p.N_pad, bp.kcb_host, kUmmaB, &b3d_host)) return DAK_ERR_CUDA;
        if (b3d_host != b3d) return DAK_ERR_CUDA;  // both maps take 64-column blocks: the same box form
    } else {
        bmap_host = bmap;
    }
    p.b3d = b3d;

    const bool pdl = t && t->pdl > 0;
    const bool fused = p.res_x || p.ss_in;
    cudaError_t e;
    if (bp.umma) {
        auto k = bp.pairs ? (fused ? gemm_umma_kernel<true, true> : gemm_umma_kernel<false, true>)
                          : (fused ? gemm_umma_kernel<true, false> : gemm_umma_kernel<false, false>);
        e = launch_ex(k, bp.grid, kUmmaThreads, bp.smem, bp.NC, pdl, stream, p, bmap, bmap_host);
    } else {
        auto k = bp.pairs ? (fused ? gemm_core_kernel<1, true, true> : gemm_core_kernel<1, false, true>)
                          : (fused ? gemm_core_kernel<1, true, false> : gemm_core_kernel<1, false, false>);
        e = launch_ex(k, bp.grid, kCoreThreads, bp.smem, 1, pdl, stream, p, bmap);
    }
    if (e == cudaSuccess && link && link->signals && p.link) *link->signals = p.n_host_ctas;
    return cuda_status(e);
}

// Any N, in column blocks of hidden-state rows (B rows and C rows of a block are
// contiguous), one launch each: by default blocks of up to kMaxWideN rows in which a
// cluster of ceil(rows / 256) CTAs shares each tile row, so the host tiles cross the link
// once per block; with column_blocks, blocks of 256 rows that each read the host tiles
// again. Clusters stop at 4 CTAs: forwarding every A chunk to 7 peers measured slower than
// two launches of 1024 rows.
static dak_status launch_gemm_column_blocks(const dak_placement* A, const void* host_src, const void* B, void* C,
                                            int N, int c_fp32, const dak_tuning* t, cudaStream_t stream, void* ws,
                                            size_t ws_bytes, const GemmFuse* fuse, const LinkHandoff* link) {
    if (link && link->signals) *link->signals = 0;
    if (!A || A->kind != 0) return DAK_ERR_INVALID;
    if (ws && (reinterpret_cast<uintptr_t>(ws) & 255)) return DAK_ERR_ALIGN;
    const int block = (t && t->column_blocks == 1) ? kMaxBlockN : kMaxWideN;
    if (N <= block) return launch_gemm_block(A, host_src, B, C, N, c_fp32, t, ws, ws_bytes, stream, fuse, link);
    if (fuse && (fuse->res_x || fuse->ss_in)) return DAK_ERR_UNSUPPORTED;
    if (!B || !C) return DAK_ERR_INVALID;
    const size_t b_row = static_cast<size_t>(A->K) * 2;
    const size_t c_row = static_cast<size_t>(A->glu ? A->M / 2 : A->M) * (c_fp32 ? 4 : 2);
    for (int n0 = 0; n0 < N; n0 += block) {
        const int nb = std::min(block, N - n0);
        const dak_status r = launch_gemm_block(A, host_src, static_cast<const uint8_t*>(B) + n0 * b_row,
                                               static_cast<uint8_t*>(C) + n0 * c_row, nb, c_fp32, t, ws, ws_bytes,
                                               stream, nullptr, nullptr);
        if (r != DAK_OK) return r;
    }
    return DAK_OK;
}

dak_status launch_gemm(const dak_placement* A, const void* host_src, const void* B, void* C, int N, int c_fp32,
                       const dak_tuning* t, cudaStream_t stream, void* ws, size_t ws_bytes, const GemmFuse* fuse,
                       const LinkHandoff* link) {
    // a public launch that joins a handoff sequence (dak_link_begin, tuning link)
    LinkHandoff own;
    int own_signals = 0;
    const bool joined = !link && link_join(t, &own);
    if (joined) {
        own.signals = &own_signals;
        link = &own;
    }
    const dak_status r = launch_gemm_column_blocks(A, host_src, B, C, N, c_fp32, t, stream, ws, ws_bytes, fuse, link);
    if (joined && r == DAK_OK) link_commit(t, own_signals);
    return r;
}


// ---------------------------------------------------------------------------------- chains
// Workspace of a chain: the operations' done counters (256 bytes), then each operation's
// per-tile-row piece counters (256-byte aligned), then each operation's partial tiles.
constexpr long long kChainDoneBytes = 256;

static long long align256(long long v) { return (v + 255) & ~255ll; }

// Plans of the chain's operations (each as a launch of its own would plan it) and the
// workspace they need; DAK_ERR_UNSUPPORTED for a chain the kernel does not take.
static dak_status plan_chain(const ChainOp* ops, int n, int N, int sms, const dak_tuning* t, BlockPlan* bps,
                             long long* cnt_off, long long* part_off, long long* need) {
    if (n < 1 || n > kMaxChainOps) return DAK_ERR_INVALID;
    if (N < 1 || N > kFuseMaxN) return DAK_ERR_UNSUPPORTED;  // tensor cores, one CTA per tile row
    long long off = kChainDoneBytes;
    for (int j = 0; j < n; ++j) {
        const dak_placement* A = ops[j].A;
        if (!A || A->kind != 0 || A->T == 0) return DAK_ERR_INVALID;
        const dak_status r = plan_block(A->T, A->h, static_cast<int>(A->K_pad), A->tile_bytes, N, sms, t, false, 0,
                                        &bps[j], A->tile_m == 2 * kTileM, 0, true);
        if (r != DAK_OK) return r;
        const BlockPlan& b = bps[j];
        if (b.pairs != bps[0].pairs) return DAK_ERR_UNSUPPORTED;  // one ring layout for every operation
        if (!b.umma || b.NC != 1 || b.kcb != b.ch[0].kc || b.ch[0].kc != b.ch[1].kc ||
            b.ch[0].stages != b.ch[1].stages || b.ch[0].stage_bytes != b.ch[1].stage_bytes)
            return DAK_ERR_UNSUPPORTED;
        if (b.ch[0].kc != bps[0].ch[0].kc || b.ch[0].stages != bps[0].ch[0].stages || b.N_pad != bps[0].N_pad)
            return DAK_ERR_UNSUPPORTED;
        cnt_off[j] = off;
        off = align256(off + static_cast<long long>(A->T) * 4);
    }
    for (int j = 0; j < n; ++j) {
        part_off[j] = off;
        if (bps[j].P > 1) off = align256(off + static_cast<long long>(ops[j].A->T + 2) * bps[j].P * kTileM * bps[j].N_pad * 4);
    }
    *need = off;
    return DAK_OK;
}

// A unit's fixed cost beside its bytes (its epilogue, the accumulator handover), in bytes
// of a CTA's stream: about half a microsecond at the per-CTA rate of a full launch.
constexpr long long kUnitFixedBytes = 32 * 1024;

// The size-balanced dealing of an independent chain all in HBM (ChainList): longest unit
// first to the CTA with the least work so far (ties: the lower CTA), each CTA's units then
// in operation order. It is taken where it cuts the busiest CTA's work (bytes plus a fixed
// cost per unit) by 3% or more against the per-operation dealing; measured on the four
// 8B-shaped linears: 74.4 -> 72.1 us at N = 32 and 83.0 -> 79.9 at N = 64, where the
// per-operation dealing leaves the busiest CTA 13% above the mean, and 0.5 us slower at
// N = 1-16, where it leaves 2%. Returns false (cl->n = 0) otherwise. The choice and the
// list are functions of the shapes and the plan only; the last ones are kept for the next
// launch.
// busiest: where given, the busiest CTA's work over the mean in thousandths, dealt per
// operation ([0]) and by size ([1]).
static bool deal_by_size(const ChainParams& cp, ChainList* cl, int* busiest = nullptr) {
    cl->n = 0;
    if (busiest) busiest[0] = busiest[1] = 0;
    const int C = cp.n_ctas;
    if (C < 1 || C > kChainListCtas) return false;
    std::vector<int> key{C, cp.n_ops};
    int total = 0;
    for (int j = 0; j < cp.n_ops; ++j) {
        const GemmParams& p = cp.op[j];
        if (p.h != 0 || cp.after_prev[j] || p.NC != 1 || p.n_hbm_ctas < 1) return false;
        total += p.gb * p.P;
        key.insert(key.end(), {p.T, p.gb, p.P, p.K_pad, p.pstep, p.pairs, p.n_host_ctas, p.n_hbm_ctas, cp.rot[j]});
    }
    if (total < 1 || total > kChainListMax) return false;
    static std::mutex mu;
    static std::vector<int> last_key;
    static ChainList last;
    static int last_busiest[2];
    std::lock_guard<std::mutex> lock(mu);
    if (key == last_key) {
        *cl = last;
        if (busiest) busiest[0] = last_busiest[0], busiest[1] = last_busiest[1];
        return cl->n > 0;
    }
    struct Unit {
        long long cost;
        int e;  // (operation << 13) | unit
    };
    std::vector<Unit> units;
    units.reserve(static_cast<size_t>(total));
    for (int j = 0; j < cp.n_ops; ++j) {
        const GemmParams& p = cp.op[j];
        const int steps = (p.K_pad + p.pstep - 1) / p.pstep;
        for (int u = 0; u < p.gb * p.P; ++u) {
            const int idx = u % p.P;
            const int k0 = (idx * steps / p.P) * p.pstep;
            const int k1 = std::min(((idx + 1) * steps / p.P) * p.pstep, p.K_pad);
            const long long bytes = static_cast<long long>(k1 - k0) * (p.pairs ? 256 : 128);
            units.push_back({bytes + kUnitFixedBytes, (j << 13) | u});
        }
    }
    // the busiest CTA under the per-operation dealing (chain_tiles without a list)
    std::vector<long long> load(static_cast<size_t>(C), 0);
    for (const Unit& x : units) {
        const GemmParams& p = cp.op[x.e >> 13];
        const int u = x.e & 0x1fff;
        load[(p.n_host_ctas + u % p.n_hbm_ctas + cp.rot[x.e >> 13]) % C] += x.cost;
    }
    const long long rr_max = *std::max_element(load.begin(), load.end());
    long long sum = 0;
    for (long long v : load) sum += v;
    std::fill(load.begin(), load.end(), 0);
    std::stable_sort(units.begin(), units.end(), [](const Unit& a, const Unit& b) { return a.cost > b.cost; });
    std::vector<std::vector<uint16_t>> per(static_cast<size_t>(C));
    for (const Unit& x : units) {
        int c = 0;
        for (int d = 1; d < C; ++d)
            if (load[d] < load[c]) c = d;
        load[c] += x.cost;
        per[c].push_back(static_cast<uint16_t>(x.e));
    }
    int at = 0;
    for (int c = 0; c < C; ++c) {
        std::sort(per[c].begin(), per[c].end());
        cl->start[c] = static_cast<uint16_t>(at);
        for (uint16_t v : per[c]) cl->e[at++] = v;
    }
    cl->start[C] = static_cast<uint16_t>(at);
    const long long size_max = *std::max_element(load.begin(), load.end());
    cl->n = size_max * 100 <= rr_max * 97 ? at : 0;
    last_key = key;
    last = *cl;
    last_busiest[0] = static_cast<int>(rr_max * 1000 * C / sum);
    last_busiest[1] = static_cast<int>(size_max * 1000 * C / sum);
    if (busiest) busiest[0] = last_busiest[0], busiest[1] = last_busiest[1];
    return cl->n > 0;
}

// The fields of a chain's parameters that its schedule and dealing read, from its plans.
static void chain_schedule(const ChainOp* ops, int n, const BlockPlan* bps, ChainParams* cp) {
    int grid = 0;
    for (int j = 0; j < n; ++j) {
        const dak_placement* A = ops[j].A;
        const BlockPlan& bp = bps[j];
        GemmParams& p = cp->op[j];
        p.K_pad = static_cast<int>(A->K_pad);
        p.NC = 1;
        p.N_pad = bp.N_pad;
        p.T = A->T;
        p.h = A->h;
        p.pairs = bp.pairs;
        p.hb = blocks_of(p.h, p.pairs);
        p.gb = blocks_of(p.T - p.h, p.pairs);
        p.P = bp.P;
        p.pstep = bp.pstep;
        p.ch[0] = bp.ch[0];
        p.ch[1] = bp.ch[1];
        p.n_host_ctas = bp.n_host_ctas;
        p.n_hbm_ctas = bp.n_hbm_ctas;
        p.host_window = p.hbm_window = bp.ch[0].stages;  // one ring for every operation
        cp->after_prev[j] = (j > 0 && ops[j].after_prev) ? 1 : 0;
        grid = std::max(grid, bp.grid);
    }
    cp->n_ops = n;
    cp->n_ctas = grid;
    // each operation starts dealing where the previous one's CTAs ended
    for (int j = 0, r = 0; j < n; ++j) {
        cp->rot[j] = r;
        r = grid > 0 ? (r + cp->op[j].n_host_ctas + cp->op[j].n_hbm_ctas) % grid : 0;
    }
}

size_t gemm_chain_workspace_bytes(const ChainOp* ops, int n, int N, const dak_tuning* t) {
    BlockPlan bps[kMaxChainOps];
    long long co[kMaxChainOps], po[kMaxChainOps], need = 0;
    if (plan_chain(ops, n, N, device_sm_count(), t, bps, co, po, &need) != DAK_OK) return 0;
    return static_cast<size_t>(need);
}

dak_status launch_gemm_chain(const ChainOp* ops, int n, int N, const dak_tuning* t, void* ws, size_t ws_bytes,
                             cudaStream_t stream) {
    if (!ops || n < 1 || n > kMaxChainOps) return DAK_ERR_INVALID;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DAK_ERR_CUDA;
    BlockPlan bps[kMaxChainOps];
    long long cnt_off[kMaxChainOps], part_off[kMaxChainOps], need = 0;
    const dak_status r = plan_chain(ops, n, N, device_sm_count(), t, bps, cnt_off, part_off, &need);
    if (r != DAK_OK) return r;
    if (!ws || static_cast<long long>(ws_bytes) < need) return DAK_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(ws) & 255) return DAK_ERR_ALIGN;

    ChainParams cp{};
    alignas(64) ChainMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    chain_schedule(ops, n, bps, &cp);
    cp.st = status_ptr();
    if (!cp.st) return DAK_ERR_CUDA;
    cp.done = static_cast<int*>(ws);
    int smem = 0;
    bool fused = false;
    for (int j = 0; j < n; ++j) {
        const ChainOp& o = ops[j];
        const dak_placement* A = o.A;
        const BlockPlan& bp = bps[j];
        if (A->device != dev) return DAK_ERR_INVALID;
        if (!o.B || !o.C) return DAK_ERR_INVALID;
        if ((reinterpret_cast<uintptr_t>(o.B) & 15) || (reinterpret_cast<uintptr_t>(o.C) & 15)) return DAK_ERR_ALIGN;
        if (A->h > 0 && !o.host_src) return DAK_ERR_INVALID;
        GemmParams& p = cp.op[j];
        p.a_host = static_cast<const uint8_t*>(o.host_src);
        p.a_hbm = static_cast<const uint8_t*>(A->hbm_ptr);
        p.B = static_cast<const __nv_bfloat16*>(o.B);
        p.C = o.C;
        p.M = static_cast<int>(A->M);
        p.K = static_cast<int>(A->K);
        p.N = N;
        p.c_fp32 = o.c_fp32 ? 1 : 0;
        p.tile_bytes = A->tile_bytes;
        p.glu = A->glu;
        p.st = cp.st;
        p.cnt = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + cnt_off[j]);
        p.part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + part_off[j]);
        const GemmFuse& f = o.fuse;
        if (f.res_x) {
            if (p.glu || o.c_fp32 || !f.res_g || !f.ss_out) return DAK_ERR_INVALID;
            p.res_x = f.res_x;
            p.res_g = static_cast<const __nv_bfloat16*>(f.res_g);
            p.ss_out = f.ss_out;
            fused = true;
        }
        if (f.ss_in) {
            if (f.ss_tiles < 1) return DAK_ERR_INVALID;
            p.ss_in = f.ss_in;
            p.ss_tiles = f.ss_tiles;
            p.ss_inv_d = f.inv_d;
            p.ss_eps = f.eps;
            fused = true;
        }
        int b3d = 0;
        if (!make_b_map(&maps.m[j], o.B, p.K, N, p.N_pad, bp.kcb, kUmmaB, &b3d)) return DAK_ERR_CUDA;
        p.b3d = b3d;
        smem = std::max(smem, bp.smem);
    }
    const int grid = cp.n_ctas;
    if (grid == 0) return DAK_OK;
    static thread_local ChainList cl;
    if (!(t && t->chain_rr > 0)) deal_by_size(cp, &cl);
    else cl.n = 0;
    auto k = fused ? gemm_chain_kernel<true> : gemm_chain_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_status(e);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(kUmmaThreads));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (t && t->pdl > 0) ? 1 : 0;
    return cuda_status(cudaLaunchKernelEx(&cfg, k, cp, maps, cl));
}

}  // namespace dak

extern "C" dak_status dak_gemm(const dak_placement* A, const void* B, void* C, int N, int c_fp32,
                               const dak_tuning* tuning, void* stream) {
    if (!A) return DAK_ERR_INVALID;
    return dak::launch_gemm(A, A->host_dev, B, C, N, c_fp32, tuning, static_cast<cudaStream_t>(stream));
}

extern "C" size_t dak_gemm_workspace_bytes(const dak_placement* A, int N) { return dak::gemm_workspace_bytes(A, N); }

static void fill_plan_info(const dak::BlockPlan& bp, int N, int block, dak_gemm_plan_info* out) {
    out->tensor_cores = bp.umma ? 1 : 0;
    out->launches = (N + block - 1) / block;
    out->cluster = bp.NC;
    out->n_pad = bp.N_pad;
    out->pieces = bp.P;
    out->piece_step = bp.pstep;
    out->chunk_k = bp.ch[0].kc;
    out->host_chunk_k = bp.ch[1].kc;
    out->hbm_stages = bp.ch[0].stages;
    out->host_stages = bp.ch[1].stages;
    out->host_ctas = bp.n_host_ctas * bp.NC;
    out->hbm_ctas = bp.n_hbm_ctas * bp.NC;
    out->host_window = bp.host_window;
    out->hbm_window = bp.hbm_window;
    out->smem_bytes = bp.smem;
    out->tile_m = bp.pairs ? 2 * dak::kTileM : dak::kTileM;
    out->cluster_slots = bp.cl_slots;
}

extern "C" dak_status dak_gemm_plan(int64_t M, int64_t K, int tile_m, int n_host_tiles, int N, int sm_count,
                                    const dak_tuning* tuning, size_t ws_bytes, dak_gemm_plan_info* out) {
    if (!out) return DAK_ERR_INVALID;
    *out = dak_gemm_plan_info{};
    if (M < 1 || K < 8 || (K % 8) || K > (1 << 24) || M > (1ll << 31) || N < 1 || sm_count < 1) return DAK_ERR_INVALID;
    if (tile_m != dak::kTileM && tile_m != 2 * dak::kTileM) return DAK_ERR_UNSUPPORTED;
    if (ws_bytes > 0 && static_cast<long long>(ws_bytes) < dak::kCallerCounterBytes) return DAK_ERR_INVALID;
    const int tiles = static_cast<int>((M + tile_m - 1) / tile_m);
    if (n_host_tiles < 0 || n_host_tiles > tiles) return DAK_ERR_INVALID;
    const int per = tile_m / dak::kTileM;  // 64-row tile rows per tile
    const int T = tiles * per;
    const int K_pad = static_cast<int>((K + 15) / 16 * 16);
    const long long tile_bytes = static_cast<long long>(dak::kTileM) * K_pad * 2;
    const int block = (tuning && tuning->column_blocks == 1) ? dak::kMaxBlockN : dak::kMaxWideN;
    dak::BlockPlan bp;
    const dak_status r = dak::plan_block(T, n_host_tiles * per, K_pad, tile_bytes, std::min(N, block), sm_count,
                                         tuning, ws_bytes > 0, ws_bytes, &bp, per == 2);
    if (r != DAK_OK) return r;
    fill_plan_info(bp, N, block, out);
    return DAK_OK;
}

extern "C" dak_status dak_gemm_chain_plan(const int64_t* M, const int64_t* K, const int* tile_m,
                                          const int* n_host_tiles, const int* after_prev, int n_ops, int N,
                                          int sm_count, const dak_tuning* tuning, dak_gemm_chain_plan_info* out) {
    if (!out) return DAK_ERR_INVALID;
    *out = dak_gemm_chain_plan_info{};
    if (!M || !K || !tile_m || !n_host_tiles || n_ops < 1 || n_ops > dak::kMaxChainOps || sm_count < 1)
        return DAK_ERR_INVALID;
    dak_placement shapes[dak::kMaxChainOps];
    dak::ChainOp ops[dak::kMaxChainOps];
    for (int j = 0; j < n_ops; ++j) {
        if (M[j] < 1 || K[j] < 8 || (K[j] % 8) || K[j] > (1 << 24) || M[j] > (1ll << 31)) return DAK_ERR_INVALID;
        if (tile_m[j] != dak::kTileM && tile_m[j] != 2 * dak::kTileM) return DAK_ERR_UNSUPPORTED;
        const int tiles = static_cast<int>((M[j] + tile_m[j] - 1) / tile_m[j]);
        if (n_host_tiles[j] < 0 || n_host_tiles[j] > tiles) return DAK_ERR_INVALID;
        const int per = tile_m[j] / dak::kTileM;
        dak_placement& A = shapes[j];
        A = dak_placement{};
        A.kind = 0;
        A.M = M[j];
        A.K = K[j];
        A.K_pad = (K[j] + 15) / 16 * 16;
        A.tile_m = tile_m[j];
        A.T = tiles * per;
        A.h = n_host_tiles[j] * per;
        A.tile_bytes = static_cast<int64_t>(dak::kTileM) * A.K_pad * 2;
        ops[j].A = &A;
        ops[j].after_prev = after_prev ? after_prev[j] : 0;
    }
    dak::BlockPlan bps[dak::kMaxChainOps];
    long long cnt_off[dak::kMaxChainOps], part_off[dak::kMaxChainOps], need = 0;
    const dak_status r = dak::plan_chain(ops, n_ops, N, sm_count, tuning, bps, cnt_off, part_off, &need);
    if (r != DAK_OK) return r;
    dak::ChainParams cp{};
    dak::chain_schedule(ops, n_ops, bps, &cp);
    static thread_local dak::ChainList cl;
    int busiest[2] = {0, 0};
    const bool by_size = dak::deal_by_size(cp, &cl, busiest);
    out->grid = cp.n_ctas;
    for (int j = 0; j < n_ops; ++j) out->units += (cp.op[j].hb + cp.op[j].gb) * cp.op[j].P;
    out->by_size = (by_size && !(tuning && tuning->chain_rr > 0)) ? 1 : 0;
    out->busiest_per_op = busiest[0];
    out->busiest_by_size = busiest[1];
    return DAK_OK;
}

extern "C" dak_status dak_gemm_launch_plan(const dak_placement* A, int N, const dak_tuning* tuning, size_t ws_bytes,
                                           dak_gemm_plan_info* out) {
    if (!A || !out || A->kind != 0 || N < 1) return DAK_ERR_INVALID;
    *out = dak_gemm_plan_info{};
    if (ws_bytes > 0 && static_cast<long long>(ws_bytes) < dak::kCallerCounterBytes) return DAK_ERR_INVALID;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DAK_ERR_CUDA;
    if (dev != A->device) return DAK_ERR_INVALID;
    const int block = (tuning && tuning->column_blocks == 1) ? dak::kMaxBlockN : dak::kMaxWideN;
    dak::BlockPlan bp;
    const dak_status r = dak::plan_launch(A, std::min(N, block), tuning, ws_bytes > 0, ws_bytes, &bp);
    if (r != DAK_OK) return r;
    fill_plan_info(bp, N, block, out);
    return DAK_OK;
}

extern "C" dak_status dak_gemm_ws(const dak_placement* A, const void* B, void* C, int N, int c_fp32,
                                  const dak_tuning* tuning, void* workspace, size_t ws_bytes, void* stream) {
    if (!A || !workspace) return DAK_ERR_INVALID;
    if (static_cast<long long>(ws_bytes) < dak::kCallerCounterBytes) return DAK_ERR_INVALID;
    return dak::launch_gemm(A, A->host_dev, B, C, N, c_fp32, tuning, static_cast<cudaStream_t>(stream), workspace,
                            ws_bytes);
}

extern "C" dak_status dak_gemm_staged(const dak_placement* A, const void* staging, const void* B, void* C, int N,
                                      int c_fp32, const dak_tuning* tuning, void* stream) {
    if (!A || (A->h > 0 && !staging)) return DAK_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(staging) & 15) return DAK_ERR_ALIGN;
    return dak::launch_gemm(A, staging, B, C, N, c_fp32, tuning, static_cast<cudaStream_t>(stream));
}

extern "C" size_t dak_gemm_chain_workspace_bytes(const dak_gemm_op* ops, int n_ops, int N, const dak_tuning* tuning) {
    if (!ops || n_ops < 1 || n_ops > dak::kMaxChainOps) return 0;
    dak::ChainOp co[dak::kMaxChainOps];
    for (int j = 0; j < n_ops; ++j) co[j].A = ops[j].A;
    return dak::gemm_chain_workspace_bytes(co, n_ops, N, tuning);
}

extern "C" dak_status dak_gemm_chain(const dak_gemm_op* ops, int n_ops, int N, const dak_tuning* tuning,
                                     void* workspace, size_t ws_bytes, void* stream) {
    if (!ops || n_ops < 1 || n_ops > dak::kMaxChainOps) return DAK_ERR_INVALID;
    dak::ChainOp co[dak::kMaxChainOps];
    for (int j = 0; j < n_ops; ++j) {
        if (!ops[j].A) return DAK_ERR_INVALID;
        co[j].A = ops[j].A;
        co[j].host_src = ops[j].A->host_dev;
        co[j].B = ops[j].B;
        co[j].C = ops[j].C;
        co[j].c_fp32 = ops[j].c_fp32;
        co[j].after_prev = ops[j].after_prev;
    }
    return dak::launch_gemm_chain(co, n_ops, N, tuning, workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}
