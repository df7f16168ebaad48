// fa_bwd.cu -- exact attention backward pass for sm_103a (GB300), behind the
// C ABI declared in include/fa.h (fa_bwd, fa_bwd_workspace_bytes).
//
// What is computed ("Why FlashAttention does not need to store the attention
// matrix", section 3.3; "CUDA FlashAttention: from online softmax to the
// long-sequence IO limit", sections 4.3.1 and 4.3.2), with dO the upstream
// gradient:
//   P     = exp(scale * Q K^T + M - LSE)   rebuilt tile by tile from the forward's LSE
//   dV    = P^T dO,   dP = dO V^T,   dS = P (x) (dP - Delta),
//   dQ    = scale * dS K,   dK = scale * dS^T Q.
// The loop order is the pages' backward order: the outer loop runs over K/V
// tiles (a work tile is 128 keys of one (b, h)), the inner loop over the Q tiles
// that see them.  dK and dV of a work tile stay on chip until it ends; dQ is
// accumulated in fp32 device memory.  Delta_i = rowsum(dP_i (x) P_i) equals
// dO_i . O_i (sum_j P_ij = 1 and O_i = sum_j P_ij v_j), which a short kernel
// computes from the forward's O before the main kernel runs.
//
// How it is computed is this file's own design for Blackwell:
//   * scores are computed transposed, S^T = K Q^T, so TMEM lane = key and
//     column = query.  The 16-bit P^T and dS^T then overwrite the fp32 S^T and
//     dP^T in place, and dV += P^T dO, dK += dS^T Q take their A operand
//     straight from TMEM;
//   * dQ^T = K^T dS^T (TMEM lane = head-dim index) reads dS^T from shared
//     memory, where the compute warps also write it in the 128-byte-swizzled
//     layout the tensor core reads.  A dQ warpgroup loads dQ^T from TMEM and
//     adds it (unscaled) into the fp32 accumulator with red.global.add, whole
//     128-byte lines per warp instruction; the final conversion applies scale;
//   * K_j and V_j are loaded once per work tile; Q_i and dO_i stream through
//     two-slot rings; LSE_i (in log2 units) and Delta_i through a two-stage
//     buffer filled by a loader warp;
//   * one warp issues every UMMA (elect.sync), two compute warpgroups each own
//     64 query columns of every key row, and the fourth warpgroup drains dQ.
// For D = 64, dQ is computed untransposed (dQ = dS K) and added row by row.
// Every mbarrier wait is bounded in time, as in the forward kernel.

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <type_traits>

#include "fa.h"
#include "fa_host.cuh"
#include "sm103_ptx.cuh"

namespace fa103 {
namespace bwd {

__device__ unsigned int g_bwd_status;

enum : unsigned {
    ST_LOAD = 1u,
    ST_MMA = 2u,
    ST_COMPUTE = 4u,
    ST_DQ = 8u,
    ST_STATS = 16u,
    ST_DRAIN = 32u,
    ST_LAYOUT = kBwdStatusLayout,
};

constexpr int kTile = 128;                    // keys of a K/V tile = query rows of a Q tile
constexpr int kThreads = 512;
constexpr uint64_t kWaitTimeoutNs = 1000000000ull;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

struct __align__(8) State {
    uint64_t kv_full, kv_empty;                 // K_j, V_j of the work tile
    uint64_t q_full[2], q_empty[2];             // Q_i ring
    uint64_t do_full[2], do_empty[2];           // dO_i ring
    uint64_t st_full[2], st_empty[2];           // LSE / Delta stages
    uint64_t s_full, dp_full;                   // S^T / dP^T of the step in TMEM (D = 128: both, on s_full)
    uint64_t p_ready;                           // P^T in TMEM (D = 64; 8 compute warps)
    uint64_t pds_ready;                         // P^T, dS^T in TMEM and dS^T in smem (8 compute warps)
    uint64_t dq_full, dq_free;                  // dQ^T in TMEM / read out (4 dQ warps)
    uint64_t dkv_full, dkv_free;                // dK, dV of the work tile complete / read out
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

template <int D>
struct Cfg {
    static constexpr int kTileBytes = kTile * D * 2;   // one 128-row tile of Q, K, V or dO
    static constexpr int kBoxes = D / 64;
    static constexpr int kBoxBytes = kTile * 128;      // 128 rows x 64 16-bit elements
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kTileBytes;
    static constexpr int kOffQ = 2 * kTileBytes;       // two slots
    static constexpr int kOffDO = 4 * kTileBytes;      // two slots
    static constexpr int kOffDS = 6 * kTileBytes;      // dS^T [key][query]: two boxes of 64 queries
    static constexpr int kOffStats = kOffDS + 2 * kBoxBytes;   // lse2[2][128], delta[2][128] fp32
    static constexpr int kOffState = kOffStats + 4 * kTile * 4;
    static constexpr int kSmemBytes = kOffState + static_cast<int>(sizeof(State));
    // Step order.  D = 64 issues S^T first and splits the compute pass: P (from
    // S^T alone) goes to TMEM and dV starts on it while dS waits for dP^T; dQ
    // then takes the dP^T / dS^T columns.  D = 128 issues dP^T first, computes P
    // and dS in one pass, and puts dQ^T over S^T / P^T (measured faster there).
    static constexpr bool kEarlyP = D == 64;
    // TMEM columns
    static constexpr uint32_t kTmA = 0;          // S^T -> P^T (16-bit) [-> dQ^T, D = 128]
    static constexpr uint32_t kTmB = 128;        // dP^T -> dS^T (16-bit) [-> dQ, D = 64]
    static constexpr uint32_t kTmDQ = kEarlyP ? kTmB : kTmA;
    static constexpr uint32_t kTmDV = 256;
    static constexpr uint32_t kTmDK = 256 + D;
};
static_assert(Cfg<128>::kSmemBytes <= 227 * 1024, "backward tiles exceed shared memory");

struct Params {
    void* dk;
    void* dv;
    float* dq_acc;        // [BH, N, D] fp32, zeroed before the main kernel
    const float* lse;     // [BH, N] natural log
    const float* delta;   // [BH, N]
    int N;
    int BH;               // query planes B * H
    int BHkv;             // K/V planes B * H_kv
    int H, H_kv;          // query heads and K/V heads per batch entry
    int G;                // H / H_kv: query heads per K/V head
    int T;                // ceil(N / 128)
    int n_tiles;          // BHkv * T
    float scale;
    float scale_log2;     // scale * log2(e)
    // Test only (fa_selftest_bwd_fault): the loader of every CTA issues no copy
    // for the Q tile of its step of this index, so the waits on it run out; -1
    // in every other launch.
    int fault_step;
};

// Work tile: K/V tile j of K/V plane kvbh.  Its steps visit Q tiles
// i0 .. T - 1 of each of the G query heads that share the K/V head, head by
// head (n_per steps each, n in all), so dK and dV sum over the group in TMEM.
struct Work {
    int kvbh, j, i0, n_per, n, qbh0;
};

template <bool CAUSAL>
__device__ __forceinline__ Work make_work(const Params& p, int idx) {
    Work w;
    w.j = idx / p.BHkv;   // j-major: under the causal mask tile j has T - j steps, heaviest first
    w.kvbh = idx - w.j * p.BHkv;
    w.i0 = CAUSAL ? w.j : 0;
    w.n_per = p.T - w.i0;
    w.n = p.G * w.n_per;
    w.qbh0 = (w.kvbh / p.H_kv) * p.H + (w.kvbh % p.H_kv) * p.G;
    return w;
}
// Q tile and query plane of the next step: Q tiles i0 .. T - 1 of one query
// head, then of the next (counters kept by each role, so no division per step).
__device__ __forceinline__ void step_next(const Work& w, int T, int& qi, int& qbh) {
    if (++qi == T) {
        qi = w.i0;
        ++qbh;
    }
}

// Work tile of this CTA's k-th turn: snake order over the CTAs.
__device__ __forceinline__ int tile_index(int k, int n_tiles) {
    const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    const long long idx = static_cast<long long>(k) * G + ((k & 1) ? (G - 1 - c) : c);
    return idx < n_tiles ? static_cast<int>(idx) : -1;
}

__device__ __forceinline__ bool wait_slow(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitTimeoutNs) return false;
    }
}
// Wait for the phase of `bar` with the given parity; false if it took longer
// than the time-out or another role gave up meanwhile.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    return mbar_try_wait(bar, parity) || wait_slow(bar, parity, abort_flag);
}
// The same by every lane of a warp, with one answer for all of them.
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag));
}

__device__ __forceinline__ void give_up(State& st, unsigned code) {
    atomicOr(&g_bwd_status, code);
    *reinterpret_cast<volatile int*>(&st.abort_flag) = 1;
}

template <int N_>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N_));
}
template <int N_>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N_));
}

__device__ __forceinline__ float bits_to_float(uint32_t h, bool bf16) {
    return bf16 ? __uint_as_float(h << 16) : __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

// ------------------------------------------------------------------ roles

// TMA producer, one thread: K_j and V_j once per work tile, then Q_i and dO_i
// of every step through their two-slot rings.
template <int D, bool CAUSAL>
__device__ void run_load(State& st, uint8_t* smem, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                         const CUtensorMap* tm_v, const CUtensorMap* tm_do, const Params& p) {
    using C = Cfg<D>;
    volatile int* abort_flag = &st.abort_flag;
    prefetch_tmap(tm_q);
    prefetch_tmap(tm_k);
    prefetch_tmap(tm_v);
    prefetch_tmap(tm_do);
    const uint64_t pol_once = l2_policy_evict_first();   // K_j, V_j: one CTA reads them
    const uint64_t pol_keep = l2_policy_evict_last();    // Q_i, dO_i: read by every K/V tile of the head
    int g = 0, kv_loads = 0;
    int q_loads[2] = {0, 0}, do_loads[2] = {0, 0};
    bool ok = true;
    for (int k = 0; ok; ++k) {
        const int idx = tile_index(k, p.n_tiles);
        if (idx < 0) break;
        const Work w = make_work<CAUSAL>(p, idx);
        if (!wait_bar(&st.kv_empty, (k & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
        }
        mbar_arrive_expect_tx(&st.kv_full, 2 * C::kTileBytes);
        for (int b = 0; b < C::kBoxes; ++b) {
            tma_load_3d_hint(smem + C::kOffK + b * C::kBoxBytes, tm_k, &st.kv_full, 64 * b, w.j * kTile, w.kvbh,
                             pol_once);
            tma_load_3d_hint(smem + C::kOffV + b * C::kBoxBytes, tm_v, &st.kv_full, 64 * b, w.j * kTile, w.kvbh,
                             pol_once);
        }
        ++kv_loads;
        int i = w.i0, qbh = w.qbh0;
        for (int s = 0; s < w.n && ok; ++s, ++g, step_next(w, p.T, i, qbh)) {
            const int slot = g & 1;
            const uint32_t ph = ((g >> 1) & 1) ^ 1;
            if (!wait_bar(&st.q_empty[slot], ph, abort_flag)) {
                ok = false;
                break;
            }
            if (g != p.fault_step) {   // test only: the fault step's Q copy is never issued
                mbar_arrive_expect_tx(&st.q_full[slot], C::kTileBytes);
                for (int b = 0; b < C::kBoxes; ++b)
                    tma_load_3d_hint(smem + C::kOffQ + slot * C::kTileBytes + b * C::kBoxBytes, tm_q,
                                     &st.q_full[slot], 64 * b, i * kTile, qbh, pol_keep);
                ++q_loads[slot];
            }
            if (!wait_bar(&st.do_empty[slot], ph, abort_flag)) {
                ok = false;
                break;
            }
            mbar_arrive_expect_tx(&st.do_full[slot], C::kTileBytes);
            for (int b = 0; b < C::kBoxes; ++b)
                tma_load_3d_hint(smem + C::kOffDO + slot * C::kTileBytes + b * C::kBoxBytes, tm_do,
                                 &st.do_full[slot], 64 * b, i * kTile, qbh, pol_keep);
            ++do_loads[slot];
        }
    }
    if (!ok) {
        give_up(st, ST_LOAD);
        // Let every copy already issued land before the CTA's shared memory goes away.
        volatile int never = 0;
        if (kv_loads > 0) wait_bar(&st.kv_full, (kv_loads - 1) & 1, &never);
        for (int s = 0; s < 2; ++s) {
            if (q_loads[s] > 0) wait_bar(&st.q_full[s], (q_loads[s] - 1) & 1, &never);
            if (do_loads[s] > 0) wait_bar(&st.do_full[s], (do_loads[s] - 1) & 1, &never);
        }
    }
}

// -LSE (converted to log2 units) and -Delta of the step's 128 query rows into a
// shared-memory stage; rows past N get LSE = +inf (so P = 0) and Delta = 0.
template <int D, bool CAUSAL>
__device__ void run_stats(State& st, uint8_t* smem, const Params& p) {
    using C = Cfg<D>;
    volatile int* abort_flag = &st.abort_flag;
    const int lane = threadIdx.x & 31;
    float* lse2s = reinterpret_cast<float*>(smem + C::kOffStats);
    float* dls = lse2s + 2 * kTile;
    int g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
        const int idx = tile_index(k, p.n_tiles);
        if (idx < 0) break;
        const Work w = make_work<CAUSAL>(p, idx);
        int qi = w.i0, qbh = w.qbh0;
        for (int s = 0; s < w.n; ++s, ++g, step_next(w, p.T, qi, qbh)) {
            const int stage = g & 1;
            ok = wait_warp(&st.st_empty[stage], ((g >> 1) & 1) ^ 1, abort_flag);
            if (!ok) break;
            const size_t rowbase = static_cast<size_t>(qbh) * p.N;
            const int q = qi * kTile + 4 * lane;
            float a[4], b[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const bool in = q + e < p.N;
                // negated, so the compute warps add them with packed FMA / add
                a[e] = in ? -(p.lse[rowbase + q + e] * kLog2e) : -INFINITY;
                b[e] = in ? -p.delta[rowbase + q + e] : 0.f;
            }
            *reinterpret_cast<float4*>(lse2s + stage * kTile + 4 * lane) = make_float4(a[0], a[1], a[2], a[3]);
            *reinterpret_cast<float4*>(dls + stage * kTile + 4 * lane) = make_float4(b[0], b[1], b[2], b[3]);
            mbar_arrive(&st.st_full[stage]);   // 32 arrivals, each releasing its own stores
        }
    }
    if (!ok && lane == 0) give_up(st, ST_STATS);
}

// UMMA issuer: warp 1, all lanes run the control flow, one elected lane issues.
// Per step: S^T = K_j Q_i^T and dP^T = V_j dO_i^T; dV += P^T dO_i once the
// compute warps have written P^T, dK += dS^T Q_i once they have written dS^T,
// then dQ^T = K_j^T dS^T (D = 128) or dQ = dS K_j (D = 64).  Cfg::kEarlyP sets
// the order of S^T and dP^T and where dQ goes in TMEM.
template <int D, bool BF16, bool CAUSAL>
__device__ void run_mma(State& st, uint8_t* smem, uint32_t tmem, const Params& p) {
    using C = Cfg<D>;
    volatile int* abort_flag = &st.abort_flag;
    const int lane = threadIdx.x & 31;
    constexpr uint32_t kIdS = idesc_f16_ab(BF16, kTile, kTile, false, false);   // S^T, dP^T
    constexpr uint32_t kIdG = idesc_f16_ab(BF16, kTile, D, false, true);        // dV, dK (A in TMEM)
    // dQ: for D = 128 as dQ^T = K^T dS^T (M = head dim, N = queries), for D = 64
    // as dQ = dS K (M = queries, N = 64): see run_dq.
    constexpr uint32_t kIdQ = D == 128 ? idesc_f16_ab(BF16, kTile, kTile, true, true)
                                       : idesc_f16_ab(BF16, kTile, D, true, true);
    const uint64_t dK = sdesc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
    const uint64_t dV = sdesc_sw128(smem_u32(smem + C::kOffV), 16, 1024);
    const uint64_t dKmn = sdesc_sw128(smem_u32(smem + C::kOffK), C::kBoxBytes, 1024);
    const uint64_t dDSmn = sdesc_sw128(smem_u32(smem + C::kOffDS), C::kBoxBytes, 1024);
    uint64_t dQk[2], dQmn[2], dDOk[2], dDOmn[2];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        dQk[s] = sdesc_sw128(smem_u32(smem + C::kOffQ + s * C::kTileBytes), 16, 1024);
        dQmn[s] = sdesc_sw128(smem_u32(smem + C::kOffQ + s * C::kTileBytes), C::kBoxBytes, 1024);
        dDOk[s] = sdesc_sw128(smem_u32(smem + C::kOffDO + s * C::kTileBytes), 16, 1024);
        dDOmn[s] = sdesc_sw128(smem_u32(smem + C::kOffDO + s * C::kTileBytes), C::kBoxBytes, 1024);
    }
    // A operand in TMEM, K-step kk over the 128 queries: P^T / dS^T of queries
    // 0..63 are at columns 0..31, of queries 64..127 at columns 64..95.
    using StepsAcol = Steps<0, 8, 16, 24, 64, 72, 80, 88>;
    using KD = typename std::conditional<D == 128, StepsK8<(C::kBoxBytes >> 4)>, StepsK4>::type;
    // S^T = K Q^T or dP^T = V dO^T: K-steps over the head dimension, both K-major
    auto issue_kd = [&](uint32_t d, uint64_t a, uint64_t b) {
        if constexpr (D == 128)
            umma_ss_x8<StepOffsets<KD, KD>>(d, a, b, kIdS, 0);
        else
            umma_ss_x4<false, StepOffsets<KD, KD>>(d, a, b, kIdS, 0);
    };

    int g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
        const int idx = tile_index(k, p.n_tiles);
        if (idx < 0) break;
        const Work w = make_work<CAUSAL>(p, idx);
        if (!wait_warp(&st.kv_full, k & 1, abort_flag) || (k > 0 && !wait_warp(&st.dkv_free, (k - 1) & 1, abort_flag))) {
            ok = false;
            break;
        }
        tc_fence_after();
        for (int s = 0; s < w.n; ++s, ++g) {
            const int slot = g & 1;
            const uint32_t ph = (g >> 1) & 1;
            if constexpr (C::kEarlyP) {
                // S^T first: its columns were last read by the previous step's dV,
                // issued before it, so it waits only for Q.
                if (!wait_warp(&st.q_full[slot], ph, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                issue_kd(tmem + C::kTmA, dK, dQk[slot]);
                umma_commit_elect(&st.s_full);
                // dP^T into the columns of the previous step's dQ, once that has been read out
                if (!wait_warp(&st.do_full[slot], ph, abort_flag) ||
                    (g > 0 && !wait_warp(&st.dq_free, (g - 1) & 1, abort_flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                issue_kd(tmem + C::kTmB, dV, dDOk[slot]);
                umma_commit_elect(&st.dp_full);
                // dV as soon as P^T is in TMEM, while the compute warps work on dS^T
                if (!wait_warp(&st.p_ready, g & 1, abort_flag)) {
                    ok = false;
                    break;
                }
            } else {
                if (!wait_warp(&st.do_full[slot], ph, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                issue_kd(tmem + C::kTmB, dV, dDOk[slot]);
                // S^T into the columns of the previous step's dQ^T, once that has been read out
                if ((g > 0 && !wait_warp(&st.dq_free, (g - 1) & 1, abort_flag)) ||
                    !wait_warp(&st.q_full[slot], ph, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                issue_kd(tmem + C::kTmA, dK, dQk[slot]);
                umma_commit_elect(&st.s_full);   // S^T and dP^T
                if (!wait_warp(&st.pds_ready, g & 1, abort_flag)) {
                    ok = false;
                    break;
                }
            }
            tc_fence_after();
            // K-step kk over the queries reads 16 rows = 2048 bytes of dO / Q (MN-major)
            umma_ts_x8<StepOffsets<StepsAcol, StepsMN8>>(tmem + C::kTmDV, tmem + C::kTmA, dDOmn[slot], kIdG,
                                                         s > 0 ? 1u : 0u);
            umma_commit_elect(&st.do_empty[slot]);
            if constexpr (C::kEarlyP) {
                if (!wait_warp(&st.pds_ready, g & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            umma_ts_x8<StepOffsets<StepsAcol, StepsMN8>>(tmem + C::kTmDK, tmem + C::kTmB, dQmn[slot], kIdG,
                                                         s > 0 ? 1u : 0u);
            umma_commit_elect(&st.q_empty[slot]);
            // dQ^T = K^T dS^T (D = 128) or dQ = dS K (D = 64), after dK (and dV) have read
            // the TMEM columns it overwrites: K-step kk over the keys reads 16 rows of K
            // and of dS^T in smem, both stored with the M or N index contiguous (MN-major)
            if constexpr (D == 128)
                umma_ss_x8<StepOffsets<StepsMN8, StepsMN8>>(tmem + C::kTmDQ, dKmn, dDSmn, kIdQ, 0);
            else
                umma_ss_x8<StepOffsets<StepsMN8, StepsMN8>>(tmem + C::kTmDQ, dDSmn, dKmn, kIdQ, 0);
            umma_commit_elect(&st.dq_full);
        }
        if (!ok) break;
        umma_commit_elect(&st.kv_empty);
        umma_commit_elect(&st.dkv_full);
    }
    if (!ok && lane == 0) give_up(st, ST_MMA);
    // Nothing of ours may still be in flight when the CTA retires.
    umma_commit_elect(&st.drain);
    volatile int never = 0;
    if (!wait_warp(&st.drain, 0, &never) && lane == 0) atomicOr(&g_bwd_status, ST_DRAIN);
}

// Compute warpgroup wg (0 or 1): TMEM lane = key row r of the work tile,
// query columns 64*wg .. 64*wg + 63 of every step, in two chunks of 32:
//   p = 2^(S^T * scale * log2 e - LSE_q * log2 e), 0 where masked,
//   ds = p (dP^T - Delta_q),
// P^T and dS^T packed to 16 bits back into TMEM, dS^T also into shared memory.
// D = 128 takes p and ds in one pass once S^T and dP^T are both in TMEM; D = 64
// first writes P^T (signalling p_ready, so dV can start) with p kept in
// registers, then waits for dP^T and writes dS^T.
// At the end of a work tile wg 0 writes the dV rows, wg 1 the dK rows.
template <int D, bool BF16, bool CAUSAL>
__device__ void run_compute(State& st, uint8_t* smem, uint32_t tmem, int wg, const Params& p) {
    using C = Cfg<D>;
    volatile int* abort_flag = &st.abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, quarter = warp & 3;
    const int r = 32 * quarter + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * quarter) << 16;
    const uint32_t tA = tmem + lane_addr + C::kTmA, tB = tmem + lane_addr + C::kTmB;
    const float* lse2s = reinterpret_cast<const float*>(smem + C::kOffStats);
    const float* dls = lse2s + 2 * kTile;
    const uint32_t ds_row = smem_u32(smem + C::kOffDS + wg * C::kBoxBytes) + static_cast<uint32_t>(r) * 128u;
    const uint32_t sw = static_cast<uint32_t>(r & 7);
    const uint64_t c2 = pack_f32x2(p.scale_log2, p.scale_log2);
    int g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
        const int idx = tile_index(k, p.n_tiles);
        if (idx < 0) break;
        const Work w = make_work<CAUSAL>(p, idx);
        const int key = w.j * kTile + r;
        const bool key_ok = key < p.N;
        int qi = w.i0, qbh = w.qbh0;
        for (int s = 0; s < w.n; ++s, ++g, step_next(w, p.T, qi, qbh)) {
            const int stage = g & 1;
            ok = wait_warp(&st.st_full[stage], (g >> 1) & 1, abort_flag) && wait_warp(&st.s_full, g & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            const bool diag = CAUSAL && qi == w.j;   // query q sees key r only if r <= q
            if constexpr (C::kEarlyP) {
                // P first, from S^T alone (dP^T may still be in the tensor core): P^T to
                // TMEM for dV, the fp32 p kept in registers for dS.
                float pk[2][32];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int col = 64 * wg + 32 * c;   // first query column of the chunk
                    uint32_t sv[32];
                    tmem_ld32_wait(tA + col, sv);
                    const float4* L = reinterpret_cast<const float4*>(lse2s + stage * kTile + col);
                    uint32_t pp[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const float4 l4 = L[e / 4];   // -LSE (log2 units)
                        float x[4];
                        unpack_f32x2(fma_f32x2(pack_f32x2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c2,
                                               pack_f32x2(l4.x, l4.y)), x[0], x[1]);
                        unpack_f32x2(fma_f32x2(pack_f32x2(__uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3])), c2,
                                               pack_f32x2(l4.z, l4.w)), x[2], x[3]);
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            float pr = ex2_approx(x[h]);
                            if (!key_ok || (diag && r > col + e + h)) pr = 0.f;
                            pk[c][e + h] = pr;
                        }
                        if constexpr (BF16) {
                            pp[e / 2] = pack_bf16x2(pk[c][e], pk[c][e + 1]);
                            pp[e / 2 + 1] = pack_bf16x2(pk[c][e + 2], pk[c][e + 3]);
                        } else {
                            pp[e / 2] = pack_f16x2(pk[c][e], pk[c][e + 1]);
                            pp[e / 2 + 1] = pack_f16x2(pk[c][e + 2], pk[c][e + 3]);
                        }
                    }
                    // P^T of these 32 queries: 16 packed columns inside the chunk's own
                    // (already read) columns -- 64*wg + 16*c is below col + 32 for c = 0 and 1.
                    tmem_st16(tA + 64 * wg + 16 * c, pp);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&st.p_ready);
                ok = wait_warp(&st.dp_full, g & 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int col = 64 * wg + 32 * c;
                    uint32_t dv[32];
                    tmem_ld32_wait(tB + col, dv);
                    const float4* Dl = reinterpret_cast<const float4*>(dls + stage * kTile + col);
                    uint32_t dd[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const float4 d4 = Dl[e / 4];   // -Delta
                        float dsv[4];
                        unpack_f32x2(mul_f32x2(pack_f32x2(pk[c][e], pk[c][e + 1]),
                                               add_f32x2(pack_f32x2(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])),
                                                         pack_f32x2(d4.x, d4.y))),
                                     dsv[0], dsv[1]);
                        unpack_f32x2(mul_f32x2(pack_f32x2(pk[c][e + 2], pk[c][e + 3]),
                                               add_f32x2(pack_f32x2(__uint_as_float(dv[e + 2]), __uint_as_float(dv[e + 3])),
                                                         pack_f32x2(d4.z, d4.w))),
                                     dsv[2], dsv[3]);
                        if constexpr (BF16) {
                            dd[e / 2] = pack_bf16x2(dsv[0], dsv[1]);
                            dd[e / 2 + 1] = pack_bf16x2(dsv[2], dsv[3]);
                        } else {
                            dd[e / 2] = pack_f16x2(dsv[0], dsv[1]);
                            dd[e / 2 + 1] = pack_f16x2(dsv[2], dsv[3]);
                        }
                    }
                    tmem_st16(tB + 64 * wg + 16 * c, dd);
                    // dS^T row r, queries 32c .. 32c+31 of box wg: 16-byte chunks 4c .. 4c+3, swizzled
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const uint32_t chunk = static_cast<uint32_t>(4 * c + cc);
                        st_shared_v4(ds_row + ((chunk ^ sw) << 4), dd[4 * cc], dd[4 * cc + 1], dd[4 * cc + 2],
                                     dd[4 * cc + 3]);
                    }
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                    const int col = 64 * wg + 32 * c;   // first query column of the chunk
                    uint32_t sv[32], dv[32];
                    tmem_ld32_nowait(tA + col, sv);
                    tmem_ld32_nowait(tB + col, dv);
                    tmem_ld_wait_regs(sv);
                    regs_after_wait(dv);
                    const float4* L = reinterpret_cast<const float4*>(lse2s + stage * kTile + col);
                    const float4* Dl = reinterpret_cast<const float4*>(dls + stage * kTile + col);
                    uint32_t pp[16], dd[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const float4 l4 = L[e / 4], d4 = Dl[e / 4];   // -LSE (log2 units), -Delta
                        float x[4], pv[4], dsv[4];
                        unpack_f32x2(fma_f32x2(pack_f32x2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c2,
                                               pack_f32x2(l4.x, l4.y)), x[0], x[1]);
                        unpack_f32x2(fma_f32x2(pack_f32x2(__uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3])), c2,
                                               pack_f32x2(l4.z, l4.w)), x[2], x[3]);
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            float pr = ex2_approx(x[h]);
                            if (!key_ok || (diag && r > col + e + h)) pr = 0.f;
                            pv[h] = pr;
                        }
                        unpack_f32x2(mul_f32x2(pack_f32x2(pv[0], pv[1]),
                                               add_f32x2(pack_f32x2(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])),
                                                         pack_f32x2(d4.x, d4.y))),
                                     dsv[0], dsv[1]);
                        unpack_f32x2(mul_f32x2(pack_f32x2(pv[2], pv[3]),
                                               add_f32x2(pack_f32x2(__uint_as_float(dv[e + 2]), __uint_as_float(dv[e + 3])),
                                                         pack_f32x2(d4.z, d4.w))),
                                     dsv[2], dsv[3]);
                        if constexpr (BF16) {
                            pp[e / 2] = pack_bf16x2(pv[0], pv[1]);
                            pp[e / 2 + 1] = pack_bf16x2(pv[2], pv[3]);
                            dd[e / 2] = pack_bf16x2(dsv[0], dsv[1]);
                            dd[e / 2 + 1] = pack_bf16x2(dsv[2], dsv[3]);
                        } else {
                            pp[e / 2] = pack_f16x2(pv[0], pv[1]);
                            pp[e / 2 + 1] = pack_f16x2(pv[2], pv[3]);
                            dd[e / 2] = pack_f16x2(dsv[0], dsv[1]);
                            dd[e / 2 + 1] = pack_f16x2(dsv[2], dsv[3]);
                        }
                    }
                    // P^T / dS^T of these 32 queries: 16 packed columns inside the chunk's own
                    // (already read) columns -- 64*wg + 16*c is below col + 32 for c = 0 and 1.
                    tmem_st16(tA + 64 * wg + 16 * c, pp);
                    tmem_st16(tB + 64 * wg + 16 * c, dd);
                    // dS^T row r, queries 32c .. 32c+31 of box wg: 16-byte chunks 4c .. 4c+3, swizzled
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const uint32_t chunk = static_cast<uint32_t>(4 * c + cc);
                        st_shared_v4(ds_row + ((chunk ^ sw) << 4), dd[4 * cc], dd[4 * cc + 1], dd[4 * cc + 2],
                                     dd[4 * cc + 3]);
                    }
                }
            }
            tmem_st_wait();
            fence_proxy_async_smem();   // dS^T in smem is read by the tensor core (async proxy)
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&st.pds_ready);
                mbar_arrive(&st.st_empty[stage]);
            }
        }
        if (!ok) break;
        // dV (wg 0) or dK (wg 1) rows of the work tile: fp32 TMEM -> 16-bit -> global
        ok = wait_warp(&st.dkv_full, k & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t tsrc = tmem + lane_addr + (wg == 0 ? C::kTmDV : C::kTmDK);
        const float mul = wg == 0 ? 1.f : p.scale;
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(wg == 0 ? p.dv : p.dk) +
                                              (static_cast<size_t>(w.kvbh) * p.N + (key_ok ? key : 0)) * D);
#pragma unroll
        for (int c = 0; c < D; c += 32) {
            uint32_t v[32];
            tmem_ld32_wait(tsrc + c, v);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float x0 = __uint_as_float(v[2 * i]) * mul, x1 = __uint_as_float(v[2 * i + 1]) * mul;
                pk[i] = BF16 ? pack_bf16x2(x0, x1) : pack_f16x2(x0, x1);
            }
            if (key_ok) {
#pragma unroll
                for (int q = 0; q < 4; ++q) dst[c / 8 + q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&st.dkv_free);
    }
    tmem_st_wait();
    if (!ok && lane == 0) give_up(st, ST_COMPUTE);
}

__device__ __forceinline__ void red_add_v2(float* addr, float a, float b) {
    asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(addr), "f"(a), "f"(b) : "memory");
}
__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// dQ warpgroup.  Per step it loads the step's dQ from TMEM, frees TMEM, then
// adds dS K (not yet multiplied by scale: the conversion kernel does that once)
// into the fp32 accumulator with red.global.add.  Measured on
// GB300, each SM's rate of writes into L2 bounds this (plain stores are hardly
// faster than reductions, and fewer CTAs reducing does not speed up the
// others), and whole 128-byte lines per warp instruction beat 16-byte pieces
// scattered over 32 rows.  So:
//   D = 128: TMEM holds dQ^T (lane = head-dim index d, column = query); a
//            2 x 2 transpose between lane pairs turns that into 8-byte
//            reductions, two whole lines (two queries) per warp instruction;
//   D = 64:  TMEM holds dQ (lane = query row, 64 columns); groups of eight
//            lanes transpose their 8 x 8 blocks of 16-byte pieces, so that a
//            16-byte reduction instruction covers four whole lines (four
//            rows) instead of pieces of 32 rows (the transposed dQ^T would
//            need M = 128 for 64 head-dim rows and leave half the lanes idle).
template <int D, bool CAUSAL>
__device__ void run_dq(State& st, uint32_t tmem, const Params& p) {
    using C = Cfg<D>;
    volatile int* abort_flag = &st.abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, quarter = warp & 3;
    // TMEM lane 32 quarter + lane: head-dim index d (D = 128) or query row (D = 64)
    const uint32_t tA = tmem + (static_cast<uint32_t>(32 * quarter) << 16) + C::kTmDQ;
    constexpr int kCols = D == 128 ? kTile : D;   // TMEM columns of the step's dQ
    int g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
        const int idx = tile_index(k, p.n_tiles);
        if (idx < 0) break;
        const Work w = make_work<CAUSAL>(p, idx);
        int qi = w.i0, qbh = w.qbh0;
        for (int s = 0; s < w.n; ++s, ++g, step_next(w, p.T, qi, qbh)) {
            ok = wait_warp(&st.dq_full, g & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            uint32_t v[kCols / 32][32];
#pragma unroll
            for (int c = 0; c < kCols / 32; ++c) tmem_ld32_nowait(tA + 32 * c, v[c]);
            tmem_ld_wait_regs(v[0]);
#pragma unroll
            for (int c = 1; c < kCols / 32; ++c) regs_after_wait(v[c]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&st.dq_free);
            const int q0 = qi * kTile;
            const size_t qplane = static_cast<size_t>(qbh) * p.N;
            if constexpr (D == 128) {
                // This thread holds dQ^T for d = 32 quarter + lane and the tile's 128
                // queries.  Lanes 2m and 2m+1 swap one value per pair of queries (a 2 x 2
                // transpose: one shuffle, three selects), after which lane 2m + b holds
                // d = 32 quarter + 2m, 2m+1 of query c + b and adds them with one 8-byte
                // reduction: a warp instruction then covers two whole 128-byte lines.
                // (A 4 x 4 transpose to 16-byte reductions, four lines per instruction,
                // costs four shuffles and sixteen selects per reduction and measured 5 %
                // slower; 4-byte reductions without a transpose, 2 % slower.)
                const int nq = p.N - q0 < kTile ? p.N - q0 : kTile;
                const int b = lane & 1;
                float* base = p.dq_acc + (qplane + q0 + b) * D + 32 * quarter + 2 * (lane >> 1);
#pragma unroll
                for (int part = 0; part < 4; ++part) {
#pragma unroll
                    for (int c0 = 0; c0 < 32; c0 += 2) {
                        const float a0 = __uint_as_float(v[part][c0]), a1 = __uint_as_float(v[part][c0 + 1]);
                        const float rcv = __shfl_xor_sync(0xffffffffu, b ? a0 : a1, 1);
                        const float x = b ? rcv : a0, y = b ? a1 : rcv;
                        const int qc = 32 * part + c0;
                        if (qc + b < nq) red_add_v2(base + static_cast<size_t>(qc) * D, x, y);
                    }
                }
            } else {
                // This thread holds the query row q0 + r (64 columns).  Per 32-column
                // half, eight lanes (eight rows) transpose their 8 x 8 block of 16-byte
                // pieces with three butterfly exchanges, after which lane 8g + b holds
                // piece b of rows 8g .. 8g+7: a warp instruction then adds four whole
                // 128-byte lines (one piece-row of four groups) instead of 32 pieces.
                const int b = lane & 7, g = lane >> 3;
                const int row0 = q0 + 32 * quarter + 8 * g;   // first row of this lane's group
                float* gbase = p.dq_acc + (qplane + row0) * D + 4 * b;
#pragma unroll
                for (int c = 0; c < kCols / 32; ++c) {
                    float a[8][4];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
#pragma unroll
                        for (int x = 0; x < 4; ++x) a[e][x] = __uint_as_float(v[c][4 * e + x]);
#pragma unroll
                    for (int d = 4; d >= 1; d >>= 1) {
                        const bool hi_lane = (lane & d) != 0;
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            if (e & d) continue;
#pragma unroll
                            for (int x = 0; x < 4; ++x) {
                                // send the piece whose bit d differs from this lane's
                                const float snd = hi_lane ? a[e][x] : a[e | d][x];
                                const float rcv = __shfl_xor_sync(0xffffffffu, snd, d);
                                if (hi_lane) a[e][x] = rcv;
                                else a[e | d][x] = rcv;
                            }
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (row0 + i < p.N)
                            red_add_v4(gbase + static_cast<size_t>(i) * D + 32 * c, a[i][0], a[i][1], a[i][2], a[i][3]);
                }
            }
        }
    }
    if (!ok && lane == 0) give_up(st, ST_DQ);
}

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const Params p) {
    using C = Cfg<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    // The swizzled tiles need 1024-byte alignment and D = 128 leaves no room to
    // realign: report and stop (uniformly, before any barrier exists).
    if (smem_u32(smem) & 1023u) {
        if (threadIdx.x == 0) atomicOr(&g_bwd_status, ST_LAYOUT);
        return;
    }
    State& st = *reinterpret_cast<State*>(smem + C::kOffState);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, wg = warp >> 2;
    if (threadIdx.x == 0) {
        mbar_init(&st.kv_full, 1);
        mbar_init(&st.kv_empty, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&st.q_full[s], 1);
            mbar_init(&st.q_empty[s], 1);
            mbar_init(&st.do_full[s], 1);
            mbar_init(&st.do_empty[s], 1);
            mbar_init(&st.st_full[s], 32);
            mbar_init(&st.st_empty[s], 8);
        }
        mbar_init(&st.s_full, 1);
        mbar_init(&st.dp_full, 1);
        mbar_init(&st.p_ready, 8);
        mbar_init(&st.pds_ready, 8);
        mbar_init(&st.dq_full, 1);
        mbar_init(&st.dq_free, 4);
        mbar_init(&st.dkv_full, 1);
        mbar_init(&st.dkv_free, 8);
        mbar_init(&st.drain, 1);
        st.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&st.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = st.tmem_base;

    // Registers: 80 + 136 + 136 + 160 = 512 per lane of a warpgroup = the launch's 128 x 512.
    if (wg == 0) {
        setmaxnreg_dec<80>();
        if (warp == 0) {
            if (lane == 0) run_load<D, CAUSAL>(st, smem, &tm_q, &tm_k, &tm_v, &tm_do, p);
            __syncwarp();
        } else if (warp == 1) {
            run_mma<D, BF16, CAUSAL>(st, smem, tmem, p);
        } else if (warp == 2) {
            run_stats<D, CAUSAL>(st, smem, p);
        }
    } else if (wg <= 2) {
        setmaxnreg_inc<136>();
        run_compute<D, BF16, CAUSAL>(st, smem, tmem, wg - 1, p);
    } else {
        setmaxnreg_inc<160>();
        run_dq<D, CAUSAL>(st, tmem, p);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Delta_i = dO_i . O_i (fp32) and the zeroed fp32 dQ accumulator row; one warp per row.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const uint16_t* __restrict__ o,
                                                         const uint16_t* __restrict__ dout, float* __restrict__ delta,
                                                         float* __restrict__ dq_acc, long long rows) {
    constexpr int kPer = D / 32;
    const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const size_t off = static_cast<size_t>(row) * D + lane * kPer;
    float acc = 0.f;
    if constexpr (kPer == 4) {
        const uint2 a = *reinterpret_cast<const uint2*>(o + off), b = *reinterpret_cast<const uint2*>(dout + off);
        const uint32_t aw[2] = {a.x, a.y}, bw[2] = {b.x, b.y};
#pragma unroll
        for (int i = 0; i < 2; ++i)
            acc += bits_to_float(aw[i] & 0xffffu, BF16) * bits_to_float(bw[i] & 0xffffu, BF16) +
                   bits_to_float(aw[i] >> 16, BF16) * bits_to_float(bw[i] >> 16, BF16);
        *reinterpret_cast<float4*>(dq_acc + off) = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
        const uint32_t a = *reinterpret_cast<const uint32_t*>(o + off), b = *reinterpret_cast<const uint32_t*>(dout + off);
        acc = bits_to_float(a & 0xffffu, BF16) * bits_to_float(b & 0xffffu, BF16) +
              bits_to_float(a >> 16, BF16) * bits_to_float(b >> 16, BF16);
        *reinterpret_cast<float2*>(dq_acc + off) = make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (lane == 0) delta[row] = acc;
}

// dQ = scale * (the fp32 accumulator of dS K) rounded to 16 bits; one warp per row.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_post_kernel(const float* __restrict__ dq_acc, uint16_t* __restrict__ dq,
                                                          long long rows, float scale) {
    constexpr int kPer = D / 32;
    const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const size_t off = static_cast<size_t>(row) * D + lane * kPer;
    if constexpr (kPer == 4) {
        float4 x = *reinterpret_cast<const float4*>(dq_acc + off);
        x.x *= scale; x.y *= scale; x.z *= scale; x.w *= scale;
        const uint2 v = BF16 ? make_uint2(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w))
                             : make_uint2(pack_f16x2(x.x, x.y), pack_f16x2(x.z, x.w));
        *reinterpret_cast<uint2*>(dq + off) = v;
    } else {
        float2 x = *reinterpret_cast<const float2*>(dq_acc + off);
        x.x *= scale; x.y *= scale;
        *reinterpret_cast<uint32_t*>(dq + off) = BF16 ? pack_bf16x2(x.x, x.y) : pack_f16x2(x.x, x.y);
    }
}

// ------------------------------------------------------------------ host

template <int D, bool BF16, bool CAUSAL>
static cudaError_t launch_main(const CUtensorMap (&m)[4], const Params& p, cudaStream_t stream) {
    auto kern = fa_bwd_kernel<D, BF16, CAUSAL>;
    static std::atomic<uint64_t> configured{0};   // one bit per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (!bit || !(configured.load() & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    const int sms = sm_count(dev);
    if (sms <= 0) return cudaErrorInvalidDevice;
    const unsigned grid = static_cast<unsigned>(p.n_tiles < sms ? p.n_tiles : sms);
    kern<<<grid, kThreads, Cfg<D>::kSmemBytes, stream>>>(m[0], m[1], m[2], m[3], p);
    return cudaGetLastError();
}

template <int D, bool BF16>
static cudaError_t launch_all(const CUtensorMap (&m)[4], const Params& p, int causal, const void* o,
                              const void* dout, void* dq, long long rows, cudaStream_t stream) {
    const unsigned grid = static_cast<unsigned>((rows + 7) / 8);
    fa_bwd_pre_kernel<D, BF16><<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(o),
                                                         static_cast<const uint16_t*>(dout),
                                                         const_cast<float*>(p.delta), p.dq_acc, rows);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = causal ? launch_main<D, BF16, true>(m, p, stream) : launch_main<D, BF16, false>(m, p, stream);
    if (e != cudaSuccess) return e;
    fa_bwd_post_kernel<D, BF16><<<grid, 256, 0, stream>>>(p.dq_acc, static_cast<uint16_t*>(dq), rows, p.scale);
    return cudaGetLastError();
}

static size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace bwd

int bwd_take_status(unsigned int* bits) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, bwd::g_bwd_status, sizeof v) != cudaSuccess) return -1;
    if (v != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(bwd::g_bwd_status, &zero, sizeof zero) != cudaSuccess) return -1;
    }
    *bits = v;
    return 0;
}

}  // namespace fa103

using namespace fa103;

extern "C" size_t fa_bwd_workspace_bytes(int B, int H, int N, int D) {
    if (B < 1 || H < 1 || N < 1 || (D != 64 && D != 128)) return 0;
    const uint64_t rows = static_cast<uint64_t>(B) * static_cast<uint64_t>(H) * static_cast<uint64_t>(N);
    if (rows * static_cast<uint64_t>(D) >= (uint64_t(1) << 40)) return 0;
    return bwd::round256(static_cast<size_t>(rows) * D * sizeof(float)) +
           bwd::round256(static_cast<size_t>(rows) * sizeof(float));
}

namespace fa103 {
namespace bwd {

// fa_bwd_gqa, with the test-only fault step of the loader (-1: none).
static int entry(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                 void* dq, void* dk, void* dv, int B, int H, int H_kv, int N, int D, float scale, int causal,
                 int dtype, void* workspace, size_t workspace_bytes, int fault_step, cudaStream_t stream) {
    if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
    if (H_kv < 1 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    const void* ptrs[10] = {q, k, v, o, dout, lse, dq, dk, dv, workspace};
    for (const void* ptr : ptrs)
        if (ptr == nullptr || (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0) return FA_ERR_MISALIGNED;
    const uint64_t BH = static_cast<uint64_t>(B) * static_cast<uint64_t>(H);
    const uint64_t BHkv = static_cast<uint64_t>(B) * static_cast<uint64_t>(H_kv);
    const uint64_t rows = BH * static_cast<uint64_t>(N);
    if (BH > 0x7fffffffull || rows * static_cast<uint64_t>(D) >= (uint64_t(1) << 40)) return FA_ERR_INVALID_ARG;
    const uint64_t T = (static_cast<uint64_t>(N) + bwd::kTile - 1) / bwd::kTile;
    if (T * BH > 0x7fffffffull) return FA_ERR_INVALID_ARG;
    const size_t need = fa_bwd_workspace_bytes(B, H, N, D);
    if (need == 0 || workspace_bytes < need) return FA_ERR_INVALID_ARG;
    const size_t tbytes = static_cast<size_t>(rows) * D * 2, lbytes = static_cast<size_t>(rows) * sizeof(float);
    const size_t kvbytes = static_cast<size_t>(BHkv * N) * D * 2;
    const void* ins[6] = {q, k, v, o, dout, lse};
    const size_t in_bytes[6] = {tbytes, kvbytes, kvbytes, tbytes, tbytes, lbytes};
    const void* outs[4] = {dq, dk, dv, workspace};
    const size_t out_bytes[4] = {tbytes, kvbytes, kvbytes, need};
    for (int a = 0; a < 4; ++a) {
        for (int b = 0; b < 6; ++b)
            if (overlaps(outs[a], out_bytes[a], ins[b], in_bytes[b])) return FA_ERR_INVALID_ARG;
        for (int b = a + 1; b < 4; ++b)
            if (overlaps(outs[a], out_bytes[a], outs[b], out_bytes[b])) return FA_ERR_INVALID_ARG;
    }
    CUtensorMap maps[4];
    const int bh = static_cast<int>(BH), bhkv = static_cast<int>(BHkv);
    if (!make_tile_map(&maps[0], q, dtype, D, N, bh) || !make_tile_map(&maps[1], k, dtype, D, N, bhkv) ||
        !make_tile_map(&maps[2], v, dtype, D, N, bhkv) || !make_tile_map(&maps[3], dout, dtype, D, N, bh))
        return FA_ERR_CUDA;
    bwd::Params p;
    p.dk = dk;
    p.dv = dv;
    p.dq_acc = static_cast<float*>(workspace);
    p.delta = reinterpret_cast<const float*>(static_cast<uint8_t*>(workspace) +
                                             bwd::round256(static_cast<size_t>(rows) * D * sizeof(float)));
    p.lse = lse;
    p.N = N;
    p.BH = bh;
    p.BHkv = bhkv;
    p.H = H;
    p.H_kv = H_kv;
    p.G = H / H_kv;
    p.T = static_cast<int>(T);
    p.n_tiles = static_cast<int>(T * BHkv);
    p.scale = scale;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.fault_step = fault_step;
    const long long nrows = static_cast<long long>(rows);
    cudaError_t e;
    if (D == 128)
        e = dtype == FA_BF16 ? bwd::launch_all<128, true>(maps, p, causal, o, dout, dq, nrows, stream)
                             : bwd::launch_all<128, false>(maps, p, causal, o, dout, dq, nrows, stream);
    else
        e = dtype == FA_BF16 ? bwd::launch_all<64, true>(maps, p, causal, o, dout, dq, nrows, stream)
                             : bwd::launch_all<64, false>(maps, p, causal, o, dout, dq, nrows, stream);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace bwd
}  // namespace fa103

extern "C" int fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dout,
                          const float* lse, void* dq, void* dk, void* dv, int B, int H, int H_kv, int N, int D,
                          float scale, int causal, int dtype, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream) {
    return bwd::entry(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, N, D, scale, causal, dtype, workspace,
                      workspace_bytes, -1, stream);
}

extern "C" int fa_selftest_bwd_fault(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                     const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int D,
                                     float scale, int causal, int dtype, void* workspace, size_t workspace_bytes,
                                     int fault_step, cudaStream_t stream) {
    if (fault_step < 0) return FA_ERR_INVALID_ARG;
    return bwd::entry(q, k, v, o, dout, lse, dq, dk, dv, B, H, H, N, D, scale, causal, dtype, workspace,
                      workspace_bytes, fault_step, stream);
}

extern "C" int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                      void* dq, void* dk, void* dv, int B, int H, int N, int D, float scale, int causal, int dtype,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return fa_bwd_gqa(q, k, v, o, dout, lse, dq, dk, dv, B, H, H, N, D, scale, causal, dtype, workspace,
                      workspace_bytes, stream);
}
