// Launch tuner: the per-operation profiling step of "DAK: Direct-Access-Enabled GPU Memory
// Offloading with Optimal Efficiency for LLM Inference", section 4.3.1 ("Congestion
// Control Strategy": how many SMs issue host requests and how many requests each keeps in
// flight are chosen per operation by measurement before launch) and section 6.2 (Fig. 12:
// congestion control and wave alignment ablations).
//
// Every candidate is timed with CUDA events over `reps` launches on a private stream after
// one warm-up launch: host CTAs x window x chunk width, then (GEMM) the pieces per tile row
// on top of the best of those. The same routine measures the two ablations: congestion
// control off (every SM may read the host tier, window 8) and wave alignment off.
#include <algorithm>
#include <vector>

#include "dak_internal.h"

namespace {

struct Timer {
    cudaStream_t s = nullptr;
    cudaEvent_t a = nullptr, b = nullptr;
    bool ok = false;
    Timer() {
        ok = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) == cudaSuccess &&
             cudaEventCreate(&a) == cudaSuccess && cudaEventCreate(&b) == cudaSuccess;
    }
    ~Timer() {
        if (a) cudaEventDestroy(a);
        if (b) cudaEventDestroy(b);
        if (s) cudaStreamDestroy(s);
    }
};

// Mean microseconds per launch of fn(tuning, stream), or a negative value if it fails.
template <typename Fn>
double time_launches(Timer& tm, Fn fn, const dak_tuning& t, int reps) {
    if (fn(&t, tm.s) != DAK_OK) return -1.0;
    if (cudaEventRecord(tm.a, tm.s) != cudaSuccess) return -1.0;
    for (int r = 0; r < reps; ++r)
        if (fn(&t, tm.s) != DAK_OK) return -1.0;
    if (cudaEventRecord(tm.b, tm.s) != cudaSuccess || cudaEventSynchronize(tm.b) != cudaSuccess) return -1.0;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, tm.a, tm.b) != cudaSuccess) return -1.0;
    return 1e3 * static_cast<double>(ms) / reps;
}

template <typename Fn>
dak_status tune(Fn fn, bool has_host, bool gemm, int reps, const dak_tuning* base, dak_tune_result* out) {
    if (!out || reps <= 0) return DAK_ERR_INVALID;
    Timer tm;
    if (!tm.ok) {
        cudaGetLastError();
        return DAK_ERR_CUDA;
    }
    dak_tuning b{};
    if (base) b = *base;
    b.link = 0;  // timed launches join no handoff sequence
    *out = dak_tune_result{};
    out->default_us = time_launches(tm, fn, b, reps);
    if (out->default_us < 0) {
        cudaGetLastError();
        return DAK_ERR_CUDA;
    }
    out->best = b;
    out->best_us = out->default_us;
    std::vector<int> hosts = has_host ? std::vector<int>{4, 8, 12, 16, 24, 32} : std::vector<int>{0};
    std::vector<int> wins = has_host ? std::vector<int>{2, 3, 4, 6, 8} : std::vector<int>{0};
    std::vector<int> chunks = gemm ? std::vector<int>{0, 256, 512} : std::vector<int>{0};
    for (int hc : hosts) {
        for (int w : wins) {
            for (int kc : chunks) {
                dak_tuning t = b;
                if (hc) t.host_ctas = hc;
                if (w) t.window = w;
                if (kc) t.chunk_k = kc;
                const double us = time_launches(tm, fn, t, reps);
                if (us < 0) {
                    cudaGetLastError();
                    continue;
                }
                ++out->candidates;
                if (us < out->best_us) {
                    out->best_us = us;
                    out->best = t;
                }
            }
        }
    }
    if (gemm && !(b.split_k > 0)) {
        // then the pieces per tile row, on top of the best host CTAs / window / chunk
        const dak_tuning top = out->best;
        for (int P : {1, 2, 3, 4, 6, 7}) {
            dak_tuning t = top;
            t.split_k = P;
            const double us = time_launches(tm, fn, t, reps);
            if (us < 0) {
                cudaGetLastError();
                continue;
            }
            ++out->candidates;
            if (us < out->best_us) {
                out->best_us = us;
                out->best = t;
            }
        }
    }
    dak_tuning off = b;
    off.host_ctas = 1 << 20;  // capped by the launcher at every slot but one
    off.window = 8;
    out->cc_off_us = has_host ? time_launches(tm, fn, off, reps) : out->default_us;
    dak_tuning na = b;
    na.no_wave_align = 1;
    out->no_align_us = time_launches(tm, fn, na, reps);
    cudaGetLastError();
    return DAK_OK;
}

}  // namespace

extern "C" dak_status dak_tune_gemm(const dak_placement* A, const void* B, void* C, int N, int c_fp32, int reps,
                                    const dak_tuning* base, dak_tune_result* out) {
    if (!A || A->kind != 0) return DAK_ERR_INVALID;
    auto fn = [&](const dak_tuning* t, cudaStream_t s) {
        return dak::launch_gemm(A, A->host_dev, B, C, N, c_fp32, t, s);
    };
    return tune(fn, A->h > 0, true, reps, base, out);
}

extern "C" dak_status dak_tune_attn(const void* Q, const dak_placement* KV, const int* seq_lens, int H_q, void* O,
                                    void* workspace, size_t ws_bytes, int reps, const dak_tuning* base,
                                    dak_tune_result* out) {
    if (!KV || KV->kind != 1) return DAK_ERR_INVALID;
    auto fn = [&](const dak_tuning* t, cudaStream_t s) {
        return dak::launch_attn(Q, KV, KV->host_dev, seq_lens, H_q, 0.f, O, workspace, ws_bytes, t, s);
    };
    return tune(fn, KV->h_s > 0, false, reps, base, out);
}
