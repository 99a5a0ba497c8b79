/*
 * dak.h -- C ABI of the direct-access tiered-memory decode library (GB300, sm_103a).
 *
 * Method: "DAK: Direct-Access-Enabled GPU Memory Offloading with Optimal Efficiency for
 * LLM Inference" (arXiv 2604.26074v1). Part of each operand lives in pinned,
 * device-mapped host memory and the rest in HBM; CTAs read each tier straight into
 * shared memory, with no staging copy in HBM (section 2.4, section 4.1).
 *
 * Conventions for every call below:
 *  - Plain pointers and sizes only. A `stream` argument is a cudaStream_t passed as
 *    void* (NULL = the legacy default stream).
 *  - Errors are returned as dak_status at once for bad arguments and launch failures;
 *    faults found on the device (a bounded wait that ran out, an index check that
 *    failed) are recorded in a device status word that dak_last_error() reads after
 *    synchronising the stream. Nothing aborts, throws or prints.
 *  - Placements (dak_placement) are owned by the library and freed by dak_free().
 *    Every other buffer (hidden states, outputs, queries, workspace) is owned by the
 *    caller and must be device memory unless stated otherwise.
 *  - All GPU work is asynchronous on `stream`. There is no CPU fallback: without a
 *    CUDA device every GPU call returns DAK_ERR_CUDA.
 */
#ifndef DAK_H
#define DAK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DAK_OK = 0,
    DAK_ERR_INVALID = 1,      /* bad argument: null pointer, size out of range, wrong placement kind */
    DAK_ERR_ALIGN = 2,        /* pointer or row pitch not 16-byte aligned, K not a multiple of 8 */
    DAK_ERR_HOST_ALLOC = 3,   /* pinned, device-mapped host allocation failed */
    DAK_ERR_DEVICE_ALLOC = 4, /* HBM allocation failed */
    DAK_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed (no device, launch error, ...) */
    DAK_ERR_TIMEOUT = 6,      /* a kernel's bounded wait ran out (reported by dak_last_error) */
    DAK_ERR_UNSUPPORTED = 7,  /* valid but not implemented shape (tile_m != 64, head dim not 64/128) */
    DAK_ERR_BOUNDS = 8        /* a kernel's index check failed (reported by dak_last_error) */
} dak_status;

const char* dak_status_string(int status);

/* Opaque, library-owned placement of one operand across the two memory tiers. */
typedef struct dak_placement dak_placement;

/* Launch tuning. Any field <= 0 takes the library default.
 *   host_ctas : CTAs that read host-resident tiles/requests; caps the number of SMs
 *               issuing host requests (section 4.3.1, "Congestion Control Strategy").
 *   window    : in-flight chunks per host CTA, the static congestion window (section 4.3.1).
 *   hbm_window: in-flight chunks per HBM CTA.
 *   chunk_k   : GEMM chunk width along K in elements (multiple of 64), the TMA chunk size
 *               exposed as a tunable in section 5 ("Cross-Architecture Adaptation").
 *   n_split   : attention context splits per (request, kv head); fixed per call and
 *               independent of the placement, so results do not depend on the offload ratio.
 *   hbm_ctas  : cap on CTAs reading HBM (0 = every remaining SM).
 *   split_k   : GEMM pieces per tile row (1..8, tensor-core path): the tile row's K range is
 *               cut at multiples of 64 columns into this many units of work that any CTA of
 *               the tile row's tier may take; the CTA that finishes a tile row's last piece
 *               adds the fp32 partials in piece order. 0 = chosen from the shape and the SM
 *               count, 1 = no split. Like chunk_k it changes the summation order, never with
 *               the offload ratio. Split launches share one device workspace: launches that
 *               split tile rows must not run concurrently on different streams.
 *   pdl       : 1 = programmatic dependent launch: the kernel may start while the previous
 *               kernel of the stream is still running; it streams the weights / KV cache at
 *               once and waits for that kernel only before reading B / Q and writing C / O.
 *               Set it only when no kernel that may still be running writes the operand
 *               being streamed or (dak_attn) seq_lens. 0 = off.
 *               2 (dak_attn only) = as 1, except that the previous kernel may write the
 *               newest token (index L_b - 1) of each request, e.g. a KV-cache append: the
 *               chunk holding it is streamed only after that kernel has finished.
 *   ctas_per_sm: dak_gemm only: size the shared-memory ring so that this many CTAs (1 or
 *               2) fit on one SM; with 2, a programmatically launched next kernel can start
 *               beside a running CTA. 0 = chosen by the library.
 *   no_wave_align: 1 = ablation of the wave alignment of section 4.1 (factor 2, Fig. 12b):
 *               host CTAs = the cap and HBM CTAs = every remaining slot, without rounding
 *               either role to whole waves. 0 = aligned (default).
 *   column_blocks: dak_gemm with N > 256 only. 0 (default) = launches of up to 1024
 *               hidden-state rows in which a cluster of ceil(rows / 256) CTAs shares each
 *               tile row: one CTA fetches every A chunk and forwards it to the others through
 *               distributed shared memory, so host bytes cross the link once per launch.
 *               1 = column blocks of 256 rows, one launch each, every block reading the
 *               host tiles again (host-link bytes = host bytes x ceil(N/256)). Like chunk_k
 *               it may change the summation order of the last, partial block (never with
 *               the offload ratio).
 *   cluster_slots: dak_gemm with N > 256: clusters the schedule assumes the GPU holds at
 *               once. 0 = asked of the device at launch (a cluster's CTAs share a GPC, so
 *               fewer clusters of 4 fit than SMs / 4; a persistent grid sized past that runs
 *               its extra clusters as a tail); dak_gemm_plan assumes sm_count / cluster.
 *   link      : dak_gemm / dak_attn: 1..8 = join host-link handoff sequence `link`, started
 *               by dak_link_begin on the same stream (see there); 0 = none. The tuner
 *               ignores it.
 *   chain_rr  : dak_gemm_chain only. 0 (default) = a chain with no tile row on the host and
 *               no after_prev deals its units (tile rows or pieces) by size: longest first
 *               to the CTA with the least work so far, so that operations of different
 *               shapes even out over the launch. 1 = every operation deals its units round
 *               the launch as its own launch would (always so for other chains). Which CTA
 *               computes a unit never changes a result.
 */
typedef struct {
    int host_ctas;
    int window;
    int hbm_window;
    int chunk_k;
    int n_split;
    int hbm_ctas;
    int split_k;
    int pdl;
    int ctas_per_sm;
    int no_wave_align;
    int column_blocks;
    int cluster_slots;
    int link;
    int chain_rr;
} dak_tuning;

/* ---------------------------------------------------------------------------------- *
 * Placement (setup, untimed)
 * ---------------------------------------------------------------------------------- */

/* Place a weight matrix A (M x K, bf16, row-major with row pitch `lda` elements) for
 * C = A x B. Section 4.1 "Data Partition" and Fig. 5a: A is cut along M into tile rows of
 * tile_m x K; tile rows 0 .. n_host_tiles-1 go to pinned, device-mapped host memory and
 * the remaining ceil(M/tile_m) - n_host_tiles rows to HBM.
 *   A_src        : source data; host memory if src_on_device == 0, else device memory.
 *                  Read once; the caller keeps ownership.
 *   tile_m       : 64 or 128 (else DAK_ERR_UNSUPPORTED). A tile is the unit of placement and
 *                  of work: 64-row tiles run M = 64 tcgen05 MMAs and spread finer over the
 *                  SMs (decode-sized N); 128-row tiles run M = 128 MMAs, about 1.7x the
 *                  tensor throughput per SM, for tensor-bound N (measured on the 8B
 *                  gate+up: 1.3x faster at N = 256, 1.75x at N = 512, all in HBM).
 *   n_host_tiles : 0 .. ceil(M/tile_m); the caller turns a ratio x into tiles (the library's
 *                  own reading is ceil(x * T)).
 * Requirements: K % 8 == 0, lda % 8 == 0, A_src 16-byte aligned (else DAK_ERR_ALIGN).
 * Internally each tier stores its tiles in a k-group-major layout ([K/8][tile_m][8]: 8 x 8
 * core blocks) that the kernels copy into shared memory with single bulk copies; a
 * 128-row tile that ends past M holds zero rows there.
 * On success *out holds a new placement (free with dak_free). Synchronous. */
dak_status dak_place_matrix(const void* A_src, int src_on_device, int64_t M, int64_t K, int64_t lda,
                            int tile_m, int n_host_tiles, dak_placement** out);

/* Place the weight of a SwiGLU projection for a fused epilogue: A_src is [2f][K] bf16 (row
 * pitch lda), the f gate rows followed by the f up rows (f a multiple of 32). The placement
 * stores them interleaved (row 2j = gate j, row 2j + 1 = up j, so every tile row holds 32
 * gate/up pairs); dak_gemm over it then writes C [N][f] = silu(gate) * up with
 * silu(z) = z / (1 + e^-z), computed in fp32 from the fp32 accumulators, instead of the
 * [N][2f] product. Otherwise as dak_place_matrix (tile rows 0 .. n_host_tiles-1 on the
 * host; 2f / 64 tile rows in all). */
dak_status dak_place_matrix_glu(const void* A_src, int src_on_device, int64_t f, int64_t K, int64_t lda, int tile_m,
                                int n_host_tiles, dak_placement** out);

/* Place a KV cache, K and V each [B][H_kv][L][D] bf16 contiguous (the pre-allocated,
 * per-request static cache of section 5). Section 5 "Supporting FlashAttention": the
 * cache is split along the batch dimension; requests 0 .. n_host_requests-1 go to pinned,
 * device-mapped host memory and the rest to HBM, so every request attends within one tier.
 * Requirements: D in {64, 128}; pointers 16-byte aligned. Synchronous. */
dak_status dak_place_kv(const void* K_src, const void* V_src, int src_on_device, int B, int H_kv, int L, int D,
                        int n_host_requests, dak_placement** out);

/* dak_place_kv at the granularity of one (request, kv head) slab: the first n_host_heads
 * slabs in request-major order (request b, head g is slab b * H_kv + g) go to the host and
 * the rest to HBM, 0 <= n_host_heads <= B * H_kv (dak_place_kv places n_host_requests *
 * H_kv). Every (request, kv head) still attends within one tier, so the attention computes
 * the same result bit for bit whatever the split; a request may now have heads in both
 * tiers. A finer unit lets a planner give the cache a ratio close to its turning point
 * when the host budget is small (one request of 16 is 6% of the cache, one slab 0.8%). */
dak_status dak_place_kv_heads(const void* K_src, const void* V_src, int src_on_device, int B, int H_kv, int L,
                              int D, int n_host_heads, dak_placement** out);

/* Append one new token to a placed KV cache (the static cache's per-step update, [DAK]
 * section 5): for every request b and kv head g, k_new[b][g][:] and v_new[b][g][:] (bf16
 * [B][H_kv][D], device, 16-byte aligned) are written at position positions[b] (int32 [B],
 * device) of that (request, kv head)'s slab, in whichever tier holds it. Stream-ordered;
 * a following dak_attn sees the token when positions[b] < its seq_lens[b] (launched with
 * tuning->pdl 2, or without programmatic launch). A position outside [0, L) is skipped and
 * reported by dak_last_error as DAK_ERR_BOUNDS. */
dak_status dak_kv_append(const dak_placement* KV, const void* k_new, const void* v_new, const int* positions,
                         void* stream);

/* Release a placement (host and HBM parts). NULL is accepted. */
dak_status dak_free(dak_placement* p);

/* Sizes of a placement: bytes in host memory and in HBM, number of units (tiles of tile_m
 * rows, or (request, kv head) slabs of a KV cache) and how many are on the host. Any
 * output pointer may be NULL. */
dak_status dak_placement_info(const dak_placement* p, int64_t* host_bytes, int64_t* hbm_bytes, int64_t* units,
                              int64_t* host_units);

/* ---------------------------------------------------------------------------------- *
 * Hot path
 * ---------------------------------------------------------------------------------- */

/* C = A x B over a tiered placement (SplitK_GEMM; section 4.1 "Kernel over Partitioned
 * Memory", "Asynchronous TMA Access", Fig. 5b).
 *   B : hidden states, bf16 [N][K] row-major (device), 16-byte aligned.
 *   C : output [N][M] row-major (device); bf16 if c_fp32 == 0, else fp32 ([N][M/2] of
 *       silu(gate) * up for a placement made by dak_place_matrix_glu).
 *   N : >= 1. Up to 256 rows run with one CTA per tile row; up to 1024 rows with a
 *       cluster of ceil(N / 256) CTAs per tile row that reads each host byte once (section
 *       4.3.2's read amplification without multicast); larger N in launches of 1024 rows
 *       (tuning->column_blocks = 1: launches of 256 rows, each re-reading the host tiles).
 * One persistent launch: `host_ctas` CTAs stream the host tile rows and the other CTAs
 * the HBM tile rows; every CTA reads from exactly one tier. When the tile rows do not
 * spread evenly over the SMs, each tile row's K range is cut into pieces (tuning split_k)
 * that the CTAs of its tier share; partial tiles go through a device workspace and the
 * CTA finishing a tile row's last piece adds them in piece order. Every output row is
 * accumulated in fp32 in an order fixed by the shape and the SM count alone, so the result
 * does not depend on n_host_tiles. N = 1 runs on CUDA cores; N >= 2 on the tcgen05 tensor
 * cores. Launches that split tile rows share the workspace: do not run them concurrently
 * on different streams of one device. */
dak_status dak_gemm(const dak_placement* A, const void* B, void* C, int N, int c_fp32, const dak_tuning* tuning,
                    void* stream);

/* dak_gemm with a split workspace of the caller's (device memory, 256-byte aligned, zeroed
 * once before its first use; dak_gemm_workspace_bytes(A, N) bytes hold every piece count a
 * launch over A with N rows may choose, 256 KiB is the least accepted). dak_gemm keeps
 * the partial tiles of split tile rows in one workspace per device, so that split
 * launches on different streams must not overlap; launches with workspaces of their own
 * may. The workspace starts with 256 KiB of per-tile-row piece counters (indexed by tile
 * row, shared by every matrix that uses the workspace) that every completed launch leaves
 * at zero; after dak_last_error reported an error, zero those 256 KiB again. The partial
 * tiles follow. A smaller workspace than a launch's pieces need makes it use fewer pieces;
 * otherwise as dak_gemm. DAK_ERR_INVALID: workspace NULL or smaller than 256 KiB;
 * DAK_ERR_ALIGN: not 256-byte aligned. */
size_t dak_gemm_workspace_bytes(const dak_placement* A, int N);
dak_status dak_gemm_ws(const dak_placement* A, const void* B, void* C, int N, int c_fp32, const dak_tuning* tuning,
                       void* workspace, size_t ws_bytes, void* stream);

/* The launch dak_gemm (ws_bytes == 0) or dak_gemm_ws (a workspace of ws_bytes) would make
 * for an M x K matrix placed in tiles of tile_m rows (64 or 128) with n_host_tiles of them
 * on the host, N hidden-state rows and the tuning, on a GPU of sm_count SMs. Host
 * arithmetic only: it needs no GPU and launches nothing. With more rows than one launch
 * takes, the fields describe the first launch. DAK_ERR_INVALID: M < 1, K not a positive
 * multiple of 8, n_host_tiles outside [0, ceil(M / tile_m)], N < 1, sm_count < 1, a non-zero
 * ws_bytes below 256 KiB, or a tuning that leaves no valid ring (e.g. chunk_k not a multiple
 * of 64); DAK_ERR_UNSUPPORTED: another tile_m. Pieces count along the K range of one tile
 * (tile_m rows). */
typedef struct {
    int tensor_cores;  /* 1: tcgen05 (N >= 2); 0: CUDA-core FMA (N == 1) */
    int launches;      /* launches (column blocks of hidden-state rows) of the call */
    int cluster;       /* CTAs per cluster that share each tile row (N > 256) */
    int n_pad;         /* hidden-state rows of one CTA's tile, padded */
    int pieces;        /* pieces each tile row's K range is cut into */
    int piece_step;    /* the pieces are cut at multiples of this many columns */
    int chunk_k;       /* columns of A per ring stage, CTAs reading HBM */
    int host_chunk_k;  /* the same for CTAs reading the host tier */
    int hbm_stages;    /* ring stages, CTAs reading HBM */
    int host_stages;   /* ring stages, CTAs reading the host tier */
    int host_ctas;     /* CTAs that stream the host tile rows */
    int hbm_ctas;      /* CTAs that stream the HBM tile rows */
    int host_window;   /* stages in flight per host CTA (congestion window) */
    int hbm_window;    /* stages in flight per HBM CTA */
    int smem_bytes;    /* dynamic shared memory per CTA */
    int tile_m;        /* tile height of the placement: 64, or 128 (M = 128 MMAs) */
    int cluster_slots; /* clusters (or CTAs, cluster == 1) the schedule counts as held at once */
} dak_gemm_plan_info;
dak_status dak_gemm_plan(int64_t M, int64_t K, int tile_m, int n_host_tiles, int N, int sm_count,
                         const dak_tuning* tuning, size_t ws_bytes, dak_gemm_plan_info* out);

/* The plan dak_gemm (ws_bytes == 0) or dak_gemm_ws would use for placement A and N
 * hidden-state rows on the current device: dak_gemm_plan's arithmetic with the device's SM
 * count and, for cluster launches, the clusters the device holds at once. Launches
 * nothing. DAK_ERR_INVALID: A not a matrix placement of this device, N < 1, ws_bytes below
 * 256 KiB but non-zero. */
dak_status dak_gemm_launch_plan(const dak_placement* A, int N, const dak_tuning* tuning, size_t ws_bytes,
                                dak_gemm_plan_info* out);

/* A chain of GEMMs C_j = A_j x B_j in one persistent launch, for 1 <= N <= 128 hidden-state
 * rows (tensor-core path; at N = 1, B padded to 8 rows as dak_gemm pads N = 2..7). The
 * paper launches one kernel per nn.Linear (section 5); here the
 * operations of a chain share one launch, so that each CTA's weight stream runs on from one
 * operation to the next instead of draining and ramping up at every launch boundary (the
 * weights never depend on an earlier operation, so a CTA streams the next operation's tiles
 * while the previous one finishes).
 *   ops[j].A, .B, .C, .c_fp32: as dak_gemm (B bf16 [N][K_j], C [N][M_j]; a placement made by
 *       dak_place_matrix_glu gives silu(gate) * up).
 *   ops[j].after_prev: 1 = operation j reads what earlier operations of the chain wrote (its B
 *       is an earlier C, or its C overwrites an earlier operation's B): its loads of B and its
 *       writes of C wait until every CTA of the launch has finished operations 0 .. j-1. 0 =
 *       independent of them (a grouped launch). ops[0].after_prev is ignored: the first
 *       operation is ordered after the previous work of the stream like any launch (with
 *       tuning->pdl, as dak_gemm with pdl).
 * Each operation is tiered, dealt to CTAs and (when its tile rows do not spread evenly) cut
 * into pieces exactly as its own dak_gemm launch would be, so results are bit-identical to
 * dak_gemm's with the same tuning, at every offload ratio (at N = 1, where dak_gemm runs on
 * the CUDA cores, they are the same product summed in another order: equal to dak_gemm to
 * fp32 rounding, and bit-identical across offload ratios). n_ops 1..8, one N for all.
 * Workspace: device memory of dak_gemm_chain_workspace_bytes(ops, n_ops, N, tuning) bytes,
 * 256-byte aligned, zeroed once before its first use: per-operation completion counters,
 * piece counters and partial tiles. Every completed launch leaves its counters at zero; after
 * dak_last_error reported an error, zero the workspace again. Launches with one workspace must
 * not overlap. The operations' completion waits are bounded (DAK_ERR_TIMEOUT through
 * dak_last_error), and every CTA of the launch must be able to run at once (the launch uses
 * at most one CTA per SM).
 * DAK_ERR_UNSUPPORTED: N outside 1..128, or operations whose launches would stream with
 * different ring layouts. DAK_ERR_INVALID: n_ops outside 1..8, null pointers, workspace
 * smaller than needed; DAK_ERR_ALIGN as dak_gemm or an unaligned workspace. */
typedef struct {
    const dak_placement* A;
    const void* B;
    void* C;
    int c_fp32;
    int after_prev;
} dak_gemm_op;
size_t dak_gemm_chain_workspace_bytes(const dak_gemm_op* ops, int n_ops, int N, const dak_tuning* tuning);
dak_status dak_gemm_chain(const dak_gemm_op* ops, int n_ops, int N, const dak_tuning* tuning, void* workspace,
                          size_t ws_bytes, void* stream);

/* How dak_gemm_chain would deal the units of a chain (its tile rows, or their pieces) over
 * its CTAs, from host arithmetic alone (no GPU): n_ops (1..8) matrices M[j] x K[j] in tiles
 * of tile_m[j] rows, n_host_tiles[j] of them on the host, after_prev[j] as in dak_gemm_op,
 * N (1..128) hidden-state rows, a GPU of sm_count SMs. A unit's work counts its bytes plus
 * 32 KiB for its fixed cost. Errors as dak_gemm_plan for each operation and as
 * dak_gemm_chain for the chain. */
typedef struct {
    int grid;            /* CTAs of the launch */
    int units;           /* units of all operations */
    int by_size;         /* 1: dealt by size (see tuning chain_rr), 0: per operation */
    int busiest_per_op;  /* the busiest CTA's work over the mean x 1000, dealt per operation */
    int busiest_by_size; /* the same dealt by size; both 0 where the size dealing does not apply
                          * (host tile rows, after_prev, more than 4096 units or 256 CTAs) */
} dak_gemm_chain_plan_info;
dak_status dak_gemm_chain_plan(const int64_t* M, const int64_t* K, const int* tile_m, const int* n_host_tiles,
                               const int* after_prev, int n_ops, int N, int sm_count, const dak_tuning* tuning,
                               dak_gemm_chain_plan_info* out);

/* Workspace bytes dak_attn needs for B requests, H_q query heads, head dim D and
 * n_split context splits (0 when n_split == 1). */
size_t dak_attn_workspace_bytes(int B, int H_q, int D, int n_split);

/* Single-query decode attention over a request-partitioned KV cache (SplitK_FlashAttn;
 * section 5). SDPA semantics for one query token per request, no mask:
 *   o[b,h] = softmax_j(scale * q[b,h] . k[b,g,j]) v[b,g,j],  g = h / (H_q / H_kv), j < L_b
 *   Q        : bf16 [B][H_q][D] (device).
 *   seq_lens : int32 [B] (device) with 1 <= L_b <= L, or NULL for all L.
 *   scale    : softmax scale; <= 0 means 1/sqrt(D).
 *   O        : bf16 [B][H_q][D] (device).
 *   workspace: device scratch of dak_attn_workspace_bytes(B, H_q, D, n_split) bytes,
 *              8-byte aligned (DAK_ERR_ALIGN otherwise; NULL allowed when that size is
 *              0), caller-owned; its contents on entry do not matter.
 * Requires H_q a multiple of H_kv with H_q / H_kv <= 16. */
dak_status dak_attn(const void* Q, const dak_placement* KV, const int* seq_lens, int H_q, float scale, void* O,
                    void* workspace, size_t ws_bytes, const dak_tuning* tuning, void* stream);

/* dak_attn with an fp32 output: O is fp32 [B][H_q][D] (device, 16-byte aligned). The parity
 * mode of the attention, as c_fp32 is dak_gemm's: scores and probabilities are fp32, and the
 * probabilities enter the P.V product as two bf16 parts (bf16(P) and bf16(P - bf16(P))), so
 * nothing on the way is rounded to bf16 except the inputs. (dak_attn feeds one bf16(P) to
 * P.V: below its bf16 output's rounding, and 4% faster on an all-HBM launch.) Arguments,
 * workspace and errors as dak_attn. */
dak_status dak_attn_f32(const void* Q, const dak_placement* KV, const int* seq_lens, int H_q, float scale, void* O,
                        void* workspace, size_t ws_bytes, const dak_tuning* tuning, void* stream);

/* The n_split dak_attn uses for a placement when tuning->n_split <= 0. */
int dak_attn_default_split(const dak_placement* KV);

/* Size of the fixed device array dak_attn_noalloc takes its workspace from: 4 MiB per
 * device (enough for B * H_q * n_split <= 8065 rows at D = 128, e.g. 32 requests x 32
 * heads x 4 splits). */
#define DAK_NOALLOC_SCRATCH_BYTES (4u << 20)

/* dak_attn for callers that cannot allocate device memory. The paper has no counterpart;
 * this is a library convenience. An engine that has already reserved the device's memory
 * for its own pools, code without access to the process's allocator, or a latency-critical
 * loop where cudaMalloc / cudaFree would synchronise the device can call this instead:
 * it allocates nothing (no cudaMalloc, cudaFree or allocating library call) and takes the
 * split workspace from a fixed array of DAK_NOALLOC_SCRATCH_BYTES compiled into the
 * library, which every device that loads the library's device code holds until exit.
 *   Arguments: as dak_attn, without workspace / ws_bytes. Q, O and seq_lens stay
 *   caller-owned device buffers.
 *   Errors: DAK_ERR_INVALID when the call would need more than DAK_NOALLOC_SCRATCH_BYTES
 *   (dak_attn_workspace_bytes(B, H_q, D, n_split) > DAK_NOALLOC_SCRATCH_BYTES); use
 *   dak_attn with a caller-provided workspace, or a smaller n_split, then.
 *   The first call on a device looks up the array's device address (cudaGetSymbolAddress,
 *   with that device current) and keeps it; make that first call before any stream
 *   capture. After cudaDeviceReset (a new context, with the array at a new address) the
 *   next call looks it up again, so make that call outside a capture too. All calls share the array and it keeps the last call's contents (nothing in
 *   it has to start at zero): calls that overlap on the GPU race on it, so order them on
 *   one stream or with events. */
dak_status dak_attn_noalloc(const void* Q, const dak_placement* KV, const int* seq_lens, int H_q, float scale,
                            void* O, const dak_tuning* tuning, void* stream);

/* ---------------------------------------------------------------------------------- *
 * Host-link handoff across launches (section 4.3.1, "Congestion Control Strategy": the
 * host requests in flight are paced; here across the operations of a step)
 * ---------------------------------------------------------------------------------- */

/* Start host-link handoff sequence `slot` (1..8) of the current device on `stream`: a
 * stream-ordered write zeroes the slot's device count, and the library's host-side count of
 * the sequence's launches restarts. Every later dak_gemm / dak_gemm_ws / dak_attn /
 * dak_attn_f32 / dak_attn_noalloc call with tuning->link = slot then joins the sequence in
 * call order: the CTAs that stream its host tiles or requests issue their first load only
 * once the host CTAs of the sequence's earlier launches have issued all of theirs, and count
 * themselves in when their own last load is issued. Under programmatic launch (tuning->pdl)
 * a launch's host CTAs otherwise fill their rings while the previous launch still streams
 * its host part, and the host link then idles through the boundary between the two; held
 * back, their loads queue right behind the previous launch's last ones. The wait is bounded
 * (0.5 ms, after which the CTA goes ahead) and only paces the loads: results never change.
 * Meant for the launches of one stream, issued (or captured into one CUDA graph) in order
 * after this call; a sequence belongs to one stream at a time. DAK_ERR_INVALID: slot out of
 * range. */
dak_status dak_link_begin(int slot, void* stream);

/* Handoff waits (of any launch, sequence or decode step) that gave up at their bound since
 * the last call: *count, after the work on `stream` has finished; the count restarts at
 * zero. A wait that gives up is no error (the CTA streams anyway and results are the
 * same), only a sign that a sequence's launches were not all ordered on one stream or
 * that an earlier launch stopped early. dak_last_error zeroes it too when it reports an
 * error. DAK_ERR_INVALID: count NULL. */
dak_status dak_link_timeouts(void* stream, uint32_t* count);

/* ---------------------------------------------------------------------------------- *
 * Launch tuner (section 4.3.1, "Congestion Control Strategy": the host-SM cap and the
 * in-flight window are profiled per operation before launch; section 6.2, Fig. 12)
 * ---------------------------------------------------------------------------------- */

/* Result of one tuning run. */
typedef struct {
    dak_tuning best;       /* fastest candidate (base with host_ctas / window / chunk_k set) */
    double best_us;        /* its mean time per launch */
    double default_us;     /* the base tuning as given */
    double cc_off_us;      /* congestion control off: every SM may read the host, window 8 */
    double no_align_us;    /* wave alignment off (no_wave_align = 1) */
    int candidates;        /* candidates timed */
} dak_tune_result;

/* Time dak_gemm(A, B, C, N, c_fp32) with `reps` launches per candidate (after one warm-up
 * launch) on a private stream, over host_ctas in {4, 8, 12, 16, 24, 32} x window in
 * {2, 3, 4, 6, 8} (when A has host tiles) x chunk_k in {library default, 256, 512}, each
 * applied on top of *base (NULL = defaults), and then, unless base fixes split_k, over
 * split_k in {1, 2, 3, 4, 6, 7} on top of the best of those; candidates the launcher
 * rejects are skipped. Synchronous; overwrites C. The chosen knobs move work between CTAs
 * only, except chunk_k and split_k, which change the summation order of every output the
 * same way at any offload ratio. */
dak_status dak_tune_gemm(const dak_placement* A, const void* B, void* C, int N, int c_fp32, int reps,
                         const dak_tuning* base, dak_tune_result* out);

/* The same for dak_attn (host_ctas x window; n_split stays base's, default when <= 0). */
dak_status dak_tune_attn(const void* Q, const dak_placement* KV, const int* seq_lens, int H_q, void* O,
                         void* workspace, size_t ws_bytes, int reps, const dak_tuning* base,
                         dak_tune_result* out);

/* ---------------------------------------------------------------------------------- *
 * Decode step of a Llama-shaped transformer around the two operations (sections 3, 5, 6.1)
 * ---------------------------------------------------------------------------------- */

/* Shape and numerics of the decoder. Fields <= 0 marked "default" take that default.
 *   n_layers, hidden (d), n_heads (H_q), n_kv_heads (H_kv), head_dim (D: 64 or 128), ffn (f).
 *   rms_eps   : RMSNorm epsilon (default 1e-5).
 *   rope_theta: RoPE base (default 500000).
 *   plain_launch: 0 = the step's kernels use programmatic dependent launch, so that each
 *               one streams its weights / KV cache while the previous one finishes;
 *               1 = ordinary stream-ordered launches.
 *   op_tuning : launch tuning of the operations qkv, o, gate_up, down (dak_gemm) and the
 *               attention (dak_attn; its n_split defaults to dak_attn_default_split of
 *               layer 0's cache), as in dak_tuning; the pdl field is set by the decoder.
 *   no_link_handoff: 0 = with programmatic launch in direct-access mode, the host tiles /
 *               requests of each operation start streaming only once the step's earlier
 *               operations have issued all their host loads, so that the host link keeps
 *               busy through the dependency at each boundary (a bounded, pacing-only wait:
 *               results are the same either way); 1 = off. */
typedef struct {
    int n_layers;
    int hidden;
    int n_heads;
    int n_kv_heads;
    int head_dim;
    int ffn;
    float rms_eps;
    float rope_theta;
    int plain_launch;
    dak_tuning op_tuning[5];
    int no_link_handoff;
} dak_decoder_config;

/* One layer's operands, all placed by the caller beforehand (dak_place_matrix with the
 * offload ratio of each operation, e.g. from dak_plan_ratios; dak_place_kv for the cache)
 * and still owned by the caller, who frees them after dak_decoder_free.
 *   qkv    : [(H_q + 2 H_kv) D] x d: query rows (head-major), then key rows, then value rows.
 *   o      : d x (H_q D).
 *   gate_up: 2f x d: the f gate rows, then the f up rows. Placed with dak_place_matrix_glu,
 *            the SwiGLU runs in the GEMM's epilogue (one launch less per layer).
 *   down   : d x f.
 *   kv     : the layer's KV cache (B requests, H_kv heads, capacity L, head dim D); every
 *            layer's cache has the same B, which is the step's batch.
 *   attn_norm, mlp_norm: RMSNorm gains, bf16 [d], device memory. */
typedef struct {
    const dak_placement* qkv;
    const dak_placement* o;
    const dak_placement* gate_up;
    const dak_placement* down;
    const dak_placement* kv;
    const void* attn_norm;
    const void* mlp_norm;
} dak_decoder_layer;

typedef struct dak_decoder dak_decoder;

/* Check the shapes, copy the layer table (not the operands) and allocate the step's
 * activations in HBM (a few MB). final_norm: bf16 [d], device. The decoder is tied to
 * the current device. */
dak_status dak_decoder_create(const dak_decoder_config* cfg, const dak_decoder_layer* layers,
                              const void* final_norm, dak_decoder** out);

/* Batch (requests per step) of a decoder: the B of its KV caches. */
int dak_decoder_batch(const dak_decoder* dec);

/* One decode step for the decoder's B requests: every layer computes
 *     h = rmsnorm(x) g_attn; [q|k|v] = h Wqkv^T; q, k = rope(q, k; pos)   (pairs i, i + D/2,
 *     angle pos * theta^(-2i/D)); append k, v to the cache at pos;
 *     x += attention(q; cache positions 0..pos) Wo^T; h = rmsnorm(x) g_mlp;
 *     x += (silu(gate) * up) Wdown^T          with [gate|up] = h Wgu^T,
 * then out = rmsnorm(x) g_final. The weight products are dak_gemm and the attention is
 * dak_attn over the tiered placements; RoPE + KV append, SwiGLU (for a placement made
 * without the gate/up interleave) and the first and last RMSNorm are small kernels of this
 * library. With B <= 128 the mid-layer RMSNorms are folded into the GEMMs around them: the
 * O and down projections add their product to x and store h = bf16(x * g) with per-64-row
 * sums of x^2, and gate+up and the next QKV multiply their fp32 accumulators by
 * 1 / sqrt(mean(x^2) + eps) (so h carries the gain but not the 1/rms factor). The residual
 * stream x is fp32; h, q, the attention output and silu(gate) * up are bf16; projections
 * accumulate in fp32.
 *   x_in     : bf16 [B][d] (device), the hidden states entering layer 0.
 *   positions: int32 [B] (device), the position of each request's new token, 0 <= pos < L
 *              (a position outside the cache is skipped and reported as DAK_ERR_BOUNDS by
 *              dak_last_error).
 *   out      : bf16 [B][d] (device).
 *   mode     : 0 = direct access (host-resident tiles and requests read in place);
 *              1 = prefetch baseline, serial: each layer's host-resident parts are first
 *                  copied into an HBM staging buffer, then the layer runs from HBM;
 *              2 = prefetch baseline, overlapped: layer l+1's copy runs on a second stream
 *                  while layer l computes (two staging buffers).
 *              Modes 1 and 2 allocate their staging buffers on first use (two buffers of
 *              the largest per-layer host bytes).
 * Only kernel launches and copies are issued on `stream` (plus the decoder's own copy
 * stream in mode 2): the call can be captured into a CUDA graph (see dak_decoder_capture),
 * once the staging buffers of modes 1 and 2 exist. */
dak_status dak_decoder_step(dak_decoder* dec, const void* x_in, const int* positions, void* out, int mode,
                            void* stream);

/* Capture one dak_decoder_step with these arguments into a CUDA graph held by the decoder
 * (replacing any earlier one). The graph reads x_in and positions and writes out at
 * replay time, so the caller refills those buffers between replays. */
dak_status dak_decoder_capture(dak_decoder* dec, const void* x_in, const int* positions, void* out, int mode);

/* Launch the captured graph on `stream`. DAK_ERR_INVALID if nothing was captured. */
dak_status dak_decoder_replay(dak_decoder* dec, void* stream);

/* Kernels one step launches in the given mode (for launch accounting). */
int dak_decoder_launches(const dak_decoder* dec, int mode);

/* Release the decoder's activations, staging buffers, streams and graph (not the
 * placements or norm gains). NULL is accepted. */
dak_status dak_decoder_free(dak_decoder* dec);

/* ---------------------------------------------------------------------------------- *
 * Planner (host only; section 4.2 and Appendix A)
 * ---------------------------------------------------------------------------------- */
typedef struct {
    double bytes;      /* C_i: bytes of weights or KV the operation reads */
    double t_comp;     /* T_comp,i: pure compute time, seconds */
    double tile_bytes; /* placement granularity in bytes (tile row or request); <= 0: continuous */
} dak_op;

/* Per-operation offload ratios minimising sum_i max(T_comp,i, (1-x_i) C_i / B_hbm,
 * x_i C_i / B_host) subject to sum_i x_i C_i >= min_offload_bytes (mode 0, the capacity
 * constraint) or == min_offload_bytes (mode 1, eq. (1) of Appendix A).
 * mode 0 and 1 solve the continuous problem with the paper's three greedy phases
 * (memory-bound operations up to their peaks, compute-bound operations up to their
 * thresholds, then any split). mode 2 solves the ">=" problem exactly over whole tiles
 * (x_i C_i a multiple of tile_bytes, capped at C_i) by dynamic programming.
 * Outputs: ratios_out[n] (x_i), model_time_out (objective, seconds; may be NULL).
 * DAK_ERR_INVALID if the budget exceeds sum C_i or an argument is out of range. */
dak_status dak_plan_ratios(const dak_op* ops, int n, double b_host, double b_hbm, double min_offload_bytes,
                           int mode, double* ratios_out, double* model_time_out);

/* Whole-unit placement for any number of operations (where the exact tile DP of mode 2 is
 * too large): ops[i].tile_bytes is operation i's placement unit (a 64-row tile row, one
 * request's KV; > 0), and it has ceil(bytes / tile_bytes) of them. The ratios of mode 0 are
 * floored to whole units; then units are added one at a time where the model time grows
 * least (ties: the operation whose ratio stays lowest) until sum_i placed bytes >=
 * min_offload_bytes. Outputs host_units_out[n] and the model time (may be NULL). */
dak_status dak_plan_units(const dak_op* ops, int n, double b_host, double b_hbm, double min_offload_bytes,
                          int64_t* host_units_out, double* model_time_out);

/* ---------------------------------------------------------------------------------- *
 * Errors, device info, measurement helpers
 * ---------------------------------------------------------------------------------- */

/* Synchronise `stream`, then read and clear the device status word. Returns DAK_OK,
 * DAK_ERR_TIMEOUT or DAK_ERR_BOUNDS (with *info, if not NULL, holding a location code). */
dak_status dak_last_error(void* stream, uint64_t* info);

/* SM count of the current device. */
int dak_sm_count(void);

/* Read-stream microbenchmark of one tier (the SM read paths the kernels use; section
 * 4.3.1 Fig. 7). Reads `bytes` from a library-allocated buffer in host memory (tier 0)
 * or HBM (tier 1) with `ctas` CTAs and `window` chunks of `chunk_bytes` in flight each,
 * `iters` times. method 0: bulk asynchronous copies into shared memory; method 1:
 * 16-byte non-coherent loads into registers; method 2: 2-D tensor-map copies.
 * Outputs the best GB/s over the iterations and whether the data read back correctly.
 * Synchronous. */
dak_status dak_probe_read_bw(int tier, int64_t bytes, int method, int ctas, int window, int chunk_bytes,
                             int iters, double* gbps_out, int* data_ok_out);

/* The congestion experiment of Fig. 7: `host_ctas` CTAs read host memory while
 * `hbm_ctas` CTAs read HBM, concurrently, with the given windows. Outputs each tier's
 * bandwidth in GB/s (bytes of that tier / that tier's busy time). Synchronous. */
dak_status dak_probe_concurrent(int64_t host_bytes, int64_t hbm_bytes, int host_ctas, int host_window,
                                int hbm_ctas, int hbm_window, int chunk_bytes, int iters, double* host_gbps,
                                double* hbm_gbps);

/* Host-side fault injection, for tests of the library's failure paths (the paper has no
 * counterpart). The library's own allocations and its tensor-map encode check a per-kind
 * switch first: after `skip` more calls of that kind succeed, the next `count` calls (-1 =
 * every call until the switch is reset) fail as if CUDA had failed, without calling it:
 *   DAK_FAULT_HOST_ALLOC   : the pinned, device-mapped host buffer of a placement or probe
 *                            (the call returns DAK_ERR_HOST_ALLOC);
 *   DAK_FAULT_DEVICE_ALLOC : the HBM part of a placement, its packing buffer, a decoder's
 *                            activations and staging, a probe's buffers (DAK_ERR_DEVICE_ALLOC);
 *   DAK_FAULT_TENSOR_MAP   : the hidden states' tensor map of dak_gemm (DAK_ERR_CUDA; nothing
 *                            is launched and C is not written).
 * A failed call frees whatever it had allocated and leaves its outputs unset. The switch is
 * process-wide. It can also be set before the process starts with the environment variable
 * DAK_FAULT_INJECT="host_alloc=SKIP:COUNT,device_alloc=COUNT,tensor_map=SKIP:COUNT" (SKIP
 * optional), read at the first allocation or fault query; dak_inject_fault overrides it.
 * DAK_ERR_INVALID for an unknown kind, skip < 0 or count < -1. Nothing touches a GPU. */
#define DAK_FAULT_HOST_ALLOC 1
#define DAK_FAULT_DEVICE_ALLOC 2
#define DAK_FAULT_TENSOR_MAP 3
dak_status dak_inject_fault(int kind, int skip, int count);

/* Injected failures of this kind still to come (-1: every call), 0 for an unknown kind. */
int dak_fault_pending(int kind);

/* Allocations the library holds right now: pinned host buffers and device buffers (each
 * placement holds at most one of each; a decoder holds its activations). For leak checks. */
dak_status dak_alloc_counts(int64_t* host_live, int64_t* device_live);

/* Self-test of the kernels' failure path: launches one CTA whose bounded wait on an
 * mbarrier that nothing arrives at runs out after about 2 s. The launch returns DAK_OK;
 * a following dak_last_error() must report DAK_ERR_TIMEOUT (info 0x5E1F in the upper 32
 * bits) and the CUDA context stays usable. The paper has no counterpart. */
dak_status dak_selftest_wait(void* stream);

/* Self-test of the handoff's pacing wait: one thread waits for a handoff count that stays
 * at zero; after 0.5 ms it gives up and goes on. Returns when the launch has finished;
 * dak_link_timeouts then reports 1 and dak_last_error DAK_OK (giving up is not an error).
 * The paper has no counterpart. */
dak_status dak_selftest_link(void* stream);

/* Prefetch baseline (section 2.2-2.3, Fig. 2-3): copy a placement's host-resident part into
 * a caller-provided HBM staging buffer (cudaMemcpyAsync on `stream`), so that a following
 * dak_gemm_staged / dak_attn_staged call reads every tile from HBM. staging must hold
 * the placement's host bytes. */
dak_status dak_prefetch(const dak_placement* p, void* staging, void* stream);

/* dak_gemm / dak_attn with the host-resident tiles or requests read from `staging`
 * (filled by dak_prefetch) instead of host memory: the all-HBM half of the prefetch
 * baseline. */
dak_status dak_gemm_staged(const dak_placement* A, const void* staging, const void* B, void* C, int N, int c_fp32,
                           const dak_tuning* tuning, void* stream);
dak_status dak_attn_staged(const void* Q, const dak_placement* KV, const void* staging, const int* seq_lens,
                           int H_q, float scale, void* O, void* workspace, size_t ws_bytes,
                           const dak_tuning* tuning, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DAK_H */
