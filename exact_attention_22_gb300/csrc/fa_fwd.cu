// fa_fwd.cu -- exact attention forward pass for sm_103a (GB300), behind the
// C ABI declared in include/fa.h.
//
// What is computed follows "CUDA FlashAttention: from online softmax to the
// long-sequence IO limit" (sections 4-6) and "Why FlashAttention does not
// need to store the attention matrix" (sections 3.2, 4.1, 4.5): per query
// row, a running max m, a running sum l and an unnormalised output O are
// carried across key/value tiles; a new tile's scores are masked (causal
// diagonal, ragged tail) before the tile max, O and l are rescaled by
// 2^(m_old - m_new) before the tile's P V is added, and the row ends with
// O / l and LSE = m + log l.  Tiles entirely above the causal diagonal are
// never visited.
//
// How it is computed is this file's own design for Blackwell:
//   * a persistent grid, one CTA per SM; a work tile is 256 query rows of one
//     (b, h) = two 128-row Q tiles ("streams" 0 and 1) that share every K/V
//     tile; tiles are dealt heaviest first, in a snake order over the CTAs;
//   * TMA loads each Q tile once and streams K_j, V_j through a shared-memory
//     ring (128-byte swizzle, mbarrier full/empty pairs);
//   * one warp issues tcgen05 UMMAs (all lanes run the control flow, one
//     elected lane issues): S_t = Q_t K_j^T into tensor memory
//     (TMEM), and O_t += P_t V_j with P_t read back from TMEM, where it
//     overwrites the first half of S_t.  When a stream finishes its K/V tiles
//     its next S is the first one of the CTA's next work tile, so the tensor
//     core keeps alternating between the streams across tile boundaries;
//   * a softmax warpgroup per stream owns one row per thread: it loads the S
//     row from TMEM, masks, takes the max, exponentiates in base 2, writes
//     P_t (16-bit) back to TMEM, and at the end of a work tile writes O / l
//     and the LSE of its rows straight from registers;
//   * a correction warpgroup rescales O_t in TMEM when a row's reference max
//     moves by more than 2^8 (the reference may lag the true max: the
//     invariant O = sum e^(s - m_ref) v, l = sum e^(s - m_ref) holds for any
//     m_ref used consistently, so the result is unchanged);
//   * with no more work tiles than SMs, a work tile is one 128-row Q tile whose
//     K/V tiles the two streams share out (key split), their partial (m, l, O)
//     merged on chip at the end of the tile.
// Every mbarrier wait is bounded in time; a wait that gives up records a
// status bit, makes the other roles stop, drains in-flight copies and MMAs,
// frees TMEM and returns.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "sm103_ptx.cuh"
#include "fa_host.cuh"

namespace fa103 {

// Status word of this library on each device: bits of the roles that gave up.
__device__ unsigned int g_fa_status;

enum : unsigned {
    ST_KV_PRODUCER = 1u,
    ST_MMA = 2u,
    ST_SOFTMAX = 4u,
    ST_CORRECTION = 8u,
    ST_DRAIN = 16u,
    ST_Q_PRODUCER = 32u,
    ST_SELFTEST = 64u,
};

constexpr int kTileM = 128;     // query rows of one Q tile (UMMA M)
constexpr int kTileN = 128;     // keys of one K/V tile (UMMA N of S, K of P V)
constexpr int kNumQ = 2;        // Q tiles (streams) per work tile
constexpr int kRowsPerTile = kTileM * kNumQ;
constexpr int kThreads = 128 * (2 + kNumQ);   // producer/MMA WG, softmax WGs, correction WG
constexpr uint64_t kWaitTimeoutNs = 1000000000ull;   // 1 s per wait
constexpr float kLazyRescale = 8.0f;          // log2 units: rescale only when the max grows > 2^8
// FP8 path: P is stored as E4M3 (largest finite 448).  A lag of the reference
// max of up to 3 log2 units and a range shift of 2^5 keep P <= 2^8, while
// probabilities down to 2^-11 stay normal numbers of the format.  (A lag of 2
// with a shift of 2^6 rescaled O more often and ran 4-7% slower.)
constexpr float kLazyRescaleFp8 = 3.0f;
constexpr float kFp8Shift = 5.0f;
constexpr float kFp8ShiftScale = 32.0f;   // 2^kFp8Shift
constexpr uint32_t kTmemCols = 512;

template <int D, bool FP8 = false>
struct Cfg {
    static constexpr int kElem = FP8 ? 1 : 2;           // bytes per element of Q, K, V
    static constexpr int kTileBytes = kTileM * D * kElem;   // one 128-row tile of Q, K or V
    static constexpr int kBoxElems = 128 / kElem;       // elements per 128-byte swizzle row
    static constexpr int kBoxes = D / kBoxElems;        // 128-byte swizzle boxes along D
    static constexpr int kBoxBytes = kTileM * 128;
    static constexpr int kStages = (D == 128 && !FP8) ? 4 : 8;  // K/V ring slots
    static constexpr int kOffQ = 0;
    static constexpr int kOffKV = kNumQ * kTileBytes;
    static constexpr int kSmemBytes = kOffKV + kStages * kTileBytes + 1024;   // + 1 KB alignment slack
    // TMEM column map: S_t (128 fp32 columns, P_t aliases its first 64), O_t (D columns)
    __host__ __device__ static constexpr uint32_t tm_s(int t) { return 128u * t; }
    __host__ __device__ static constexpr uint32_t tm_o(int t) { return 256u + static_cast<uint32_t>(D) * t; }
};

struct __align__(8) SharedState {
    uint64_t q_full[kNumQ];        // Q producer -> MMA: Q_t of the current work tile landed
    uint64_t q_empty[kNumQ];       // MMA -> Q producer: the last S_t of a work tile finished
    uint64_t kv_full[8];
    uint64_t kv_empty[8];
    uint64_t s_full[kNumQ];        // MMA -> softmax: S_t of the current step is in TMEM
    uint64_t p_full[kNumQ];        // softmax + correction -> MMA: P_t in TMEM and O_t rescaled
    uint64_t alpha_ready[kNumQ];   // softmax -> correction: per-row rescale factors published
    uint64_t pv_done[kNumQ];       // MMA -> softmax/correction: O_t += P_t V_j complete
    uint64_t k_sync[4];            // key split: both streams' warps of one TMEM lane quarter
    uint64_t drain;
    float alpha[kNumQ][kTileM];
    float4 k_part[kNumQ][kTileM];  // key split: each stream's (m_ref, l, ls) of a row
    uint32_t tmem_base;
    int abort_flag;
};

struct Params {
    void* o;
    float* lse;
    float* ws_o;         // split mode: partial O, [splits][BH][N][D] fp32 (null otherwise)
    float4* ws_st;       // split mode: partial (m, l, l_exact, -), [splits][BH][N]
    int N;               // query rows of a Q plane (the sequence length for square attention)
    int Nk;              // keys of a K/V plane
    int q_per;           // query positions per head (rows of a plane are q_per x heads when packed)
    int causal_off;      // Nk - q_per: query position i is the token at i + causal_off
    int packed;          // 1: a Q plane stacks the query heads that share one K/V head
    int BH;
    int H;               // query heads per batch entry
    int kv_group;        // query heads per K/V head (1 without grouped K/V heads)
    int n_qblocks;       // ceil(N / 256)
    int n_splits;        // chunks of K/V tiles per query block (1 without a split)
    int n_tiles;         // n_qblocks * BH * n_splits
    float scale_log2;    // scale * log2(e)
    // FP8 path: per-block dequantization scales [BH][n_blocks] of Q, K and V
    // (K and V indexed by the K/V head), 128 rows (keys) per block.
    const float* q_scale;
    const float* k_scale;
    const float* v_scale;
    int n_blocks;
    // Test only (fa_selftest_fwd_fault): the K/V producer of every CTA issues
    // no copy for its ring item of this index, so the waits on it run out; -1
    // in every other launch.
    int fault_item;
};

// One work tile: query rows q0 .. q0+255 of head bh, K/V tiles j0 .. j0+n_all-1
// (chunk `split` of the query block's range).  In the key-split form (below):
// query rows q0 .. q0+127 for both streams, stream 0 on K/V tiles 0 .. nkv[0]-1
// and stream 1 on j0 .. j0+nkv[1]-1.
struct Tile {
    int q0, bh, kvh, split, j0, n_all;   // kvh: K/V plane b * H_kv + h / kv_group
    int nkv[kNumQ];      // K/V tiles of this chunk each stream visits (0: none)
};

// Key-split work tiles (KS, few work tiles for the SMs): one 128-row Q tile of
// one plane; both streams take its rows, stream 0 the first ceil(J/2) of its J
// K/V tiles and stream 1 the rest (starting at tile j0), and the two partial
// (m, l, O) are merged at the end of the tile.
template <bool CAUSAL>
__device__ __forceinline__ Tile make_tile_ks(const Params& p, int idx) {
    Tile w;
    w.split = 0;
    w.q0 = (p.n_qblocks - 1 - idx / p.BH) * kTileM;   // heaviest first
    w.bh = idx % p.BH;
    w.kvh = p.kv_group == 1 ? w.bh : (w.bh / p.H) * (p.H / p.kv_group) + (w.bh % p.H) / p.kv_group;
    int J;
    if (CAUSAL) {
        const int qlast = min(w.q0 + kTileM - 1, p.N - 1);
        J = qlast + p.causal_off < 0 ? 0 : min(qlast + p.causal_off, p.Nk - 1) / kTileN + 1;
    } else {
        J = (p.Nk + kTileN - 1) / kTileN;
    }
    w.nkv[0] = (J + 1) / 2;
    w.nkv[1] = J / 2;
    w.j0 = w.nkv[0];
    w.n_all = w.nkv[0];
    return w;
}

template <bool CAUSAL, bool SPLIT, bool KS = false>
__device__ __forceinline__ Tile make_tile(const Params& p, int idx) {
    if constexpr (KS) return make_tile_ks<CAUSAL>(p, idx);
    Tile w;
    // heaviest query block first: causal work grows with the block index
    const int qbh = SPLIT ? idx / p.n_splits : idx;
    w.split = SPLIT ? idx - qbh * p.n_splits : 0;
    w.q0 = (p.n_qblocks - 1 - qbh / p.BH) * kRowsPerTile;
    w.bh = qbh % p.BH;
    w.kvh = p.kv_group == 1 ? w.bh : (w.bh / p.H) * (p.H / p.kv_group) + (w.bh % p.H) / p.kv_group;
    int full[kNumQ], full_all = 0;
#pragma unroll
    for (int t = 0; t < kNumQ; ++t) {
        const int r0 = w.q0 + kTileM * t;
        if (r0 >= p.N) {
            full[t] = 0;
        } else if (CAUSAL) {
            // the last key any row of this Q tile sees: that of its last position
            const int qlast = p.packed ? p.q_per - 1 : min(r0 + kTileM - 1, p.N - 1);
            full[t] = min(qlast + p.causal_off, p.Nk - 1) / kTileN + 1;
        } else {
            full[t] = (p.Nk + kTileN - 1) / kTileN;
        }
        full_all = max(full_all, full[t]);
    }
    // chunk `split` of the query block's K/V range [0, full_all)
    const int chunk = SPLIT ? (full_all + p.n_splits - 1) / p.n_splits : full_all;
    w.j0 = SPLIT ? min(w.split * chunk, full_all) : 0;
    const int j1 = SPLIT ? min(w.j0 + chunk, full_all) : full_all;
    w.n_all = 0;
#pragma unroll
    for (int t = 0; t < kNumQ; ++t) {
        w.nkv[t] = max(0, min(j1, full[t]) - w.j0);
        w.n_all = max(w.n_all, w.nkv[t]);
    }
    return w;
}

// First query row of stream t's Q tile, and its first K/V tile.
template <bool KS>
__device__ __forceinline__ int stream_row0(const Tile& w, int t) { return KS ? w.q0 : w.q0 + kTileM * t; }
template <bool KS>
__device__ __forceinline__ int stream_kv0(const Tile& w, int t) { return KS ? (t ? w.j0 : 0) : w.j0; }

// The k-th work tile of this CTA, or -1: rounds of gridDim.x tiles, dealt in a
// snake order so a CTA that got a heavy tile in one round gets a light one in
// the next.
__device__ __forceinline__ int tile_index(int k, int n_tiles) {
    const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    const long long idx = static_cast<long long>(k) * G + ((k & 1) ? (G - 1 - c) : c);
    return idx < n_tiles ? static_cast<int>(idx) : -1;
}

__device__ __forceinline__ bool wait_bar_slow(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
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
    return mbar_try_wait(bar, parity) || wait_bar_slow(bar, parity, abort_flag);
}

__device__ __forceinline__ void give_up(SharedState& sh, unsigned code) {
    atomicOr(&g_fa_status, code);
    *reinterpret_cast<volatile int*>(&sh.abort_flag) = 1;
}

template <int N_>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N_));
}
template <int N_>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N_));
}

// 128 consecutive TMEM columns of this thread's lane, one wait for both loads.
__device__ __forceinline__ void tmem_ld128_wait(uint32_t taddr, float (&s)[128]) {
    uint32_t(&r)[128] = reinterpret_cast<uint32_t(&)[128]>(s);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
        "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%128];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
        "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,"
        "%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,"
        "%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%129];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]),
          "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]),
          "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]),
          "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]),
          "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]),
          "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]),
          "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]),
          "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]),
          "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]),
          "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]),
          "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]),
          "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]),
          "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]),
          "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]),
          "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
        : "r"(taddr), "r"(taddr + 64)
        : "memory");
}

// ------------------------------------------------------------------ roles

// K/V producer: one thread; K_j then V_j of every work tile, in order.
template <int D, bool CAUSAL, bool SPLIT, bool FP8, bool KS>
__device__ void run_kv_producer(SharedState& sh, uint8_t* tiles, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                const Params& p) {
    using C = Cfg<D, FP8>;
    volatile int* abort_flag = &sh.abort_flag;
    prefetch_tmap(tm_k);
    prefetch_tmap(tm_v);
    const uint64_t pol_keep = l2_policy_evict_last();   // K, V: re-read by the head's other work tiles
    int item = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
        const int idx = tile_index(k, p.n_tiles);
        if (idx < 0) break;
        const Tile w = make_tile<CAUSAL, SPLIT, KS>(p, idx);
        for (int j = 0; j < w.n_all && ok; ++j)
#pragma unroll 1
        for (int t = 0; t < (KS ? kNumQ : 1) && ok; ++t) {
            // key split: stream 0's j-th K/V tile, then stream 1's (if it has one)
            if (KS && j >= w.nkv[t]) continue;
            const int jt = stream_kv0<KS>(w, t) + j;
#pragma unroll 1
            for (int kind = 0; kind < 2; ++kind, ++item) {   // K_j, then V_j
                const int slot = item % C::kStages;
                if (!wait_bar(&sh.kv_empty[slot], ((item / C::kStages) & 1) ^ 1, abort_flag)) {
                    give_up(sh, ST_KV_PRODUCER);
                    ok = false;
                    break;
                }
                if (item == p.fault_item) continue;   // test only: this copy is never issued
                mbar_arrive_expect_tx(&sh.kv_full[slot], C::kTileBytes);
                const CUtensorMap* map = kind ? tm_v : tm_k;
                uint8_t* dst = tiles + C::kOffKV + slot * C::kTileBytes;
                if (FP8 && kind) {
                    // V is stored transposed per head ([D][N], keys contiguous): one
                    // 128-key x 128-row box, the operand K-major for the FP8 P V
                    tma_load_3d_hint(dst, map, &sh.kv_full[slot], jt * kTileN, 0, w.kvh, pol_keep);
                } else {
                    for (int b = 0; b < C::kBoxes; ++b)
                        tma_load_3d_hint(dst + b * C::kBoxBytes, map, &sh.kv_full[slot], C::kBoxElems * b,
                                         jt * kTileN, w.kvh, pol_keep);
                }
            }
        }
    }
    if (!ok) {
        // Let every copy already issued (items < item) land before the CTA's
        // shared memory goes away: the last item of each slot is enough.
        volatile int never = 0;
        for (int last = item - 1; last >= 0 && last >= item - C::kStages; --last)
            if (last != p.fault_item) wait_bar(&sh.kv_full[last % C::kStages], (last / C::kStages) & 1, &never);
    }
}

// Q producer: one thread; Q_t of every work tile once its buffer is free.
template <int D, bool CAUSAL, bool SPLIT, bool FP8, bool KS>
__device__ void run_q_producer(SharedState& sh, uint8_t* tiles, const CUtensorMap* tm_q, const Params& p) {
    using C = Cfg<D, FP8>;
    volatile int* abort_flag = &sh.abort_flag;
    prefetch_tmap(tm_q);
    const uint64_t pol_once = l2_policy_evict_first();   // Q: read once
    int loads[kNumQ] = {0, 0};
    bool ok = true;
    for (int k = 0; ok; ++k) {
        const int idx = tile_index(k, p.n_tiles);
        if (idx < 0) break;
        const Tile w = make_tile<CAUSAL, SPLIT, KS>(p, idx);
        for (int t = 0; t < kNumQ; ++t) {
            if (w.nkv[t] == 0) continue;
            if (!wait_bar(&sh.q_empty[t], (loads[t] & 1) ^ 1, abort_flag)) {
                give_up(sh, ST_Q_PRODUCER);
                ok = false;
                break;
            }
            mbar_arrive_expect_tx(&sh.q_full[t], C::kTileBytes);
            for (int b = 0; b < C::kBoxes; ++b)
                tma_load_3d_hint(tiles + C::kOffQ + t * C::kTileBytes + b * C::kBoxBytes, tm_q, &sh.q_full[t],
                                 C::kBoxElems * b, stream_row0<KS>(w, t), w.bh, pol_once);
            ++loads[t];
        }
    }
    if (!ok) {
        volatile int never = 0;
        for (int t = 0; t < kNumQ; ++t)
            if (loads[t] > 0) wait_bar(&sh.q_full[t], (loads[t] - 1) & 1, &never);
    }
}

__device__ __forceinline__ int lane_id() { return static_cast<int>(threadIdx.x & 31); }
// Three barrier tests by lane 0, result broadcast so the warp stays uniform.
__device__ __forceinline__ uint32_t mbar_test3_bcast(uint64_t* b0, uint32_t p0, uint64_t* b1, uint32_t p1, uint64_t* b2,
                                                     uint32_t p2) {
    return __shfl_sync(0xffffffffu, mbar_test3(b0, p0, b1, p1, b2, p2), 0);
}

// UMMA issuer: warp 1.  All 32 lanes run the control flow below with the same
// values, and each tcgen05.mma / tcgen05.commit is issued by one elected lane.
//
// Ring items are K_0, V_0, K_1, V_1, ... of each work tile in turn; they are
// acquired (full barrier waited) in that order.  An item is released (its
// slot's empty barrier committed after the MMA that reads it) by the last
// MMA issued that reads it.  Within a round stream 0 goes first, so that is
// stream 1 where it reads the item, else stream 0.  The one exception is a
// work tile's K_0: a stream's first S of the next tile goes out early, at the
// end of its previous tile, and stream 0 may start only at the top of the tile
// (when it had no K/V tiles in the previous one), after stream 1.
template <int D, bool BF16, bool CAUSAL, bool SPLIT, bool FP8, bool KS>
__device__ void run_mma(SharedState& sh, uint8_t* tiles, uint32_t tmem, const Params& p) {
    using C = Cfg<D, FP8>;
    volatile int* abort_flag = &sh.abort_flag;
    // FP8: kind::f8f6f4 with E4M3 operands (format code 0 in the A / B fields);
    // P V then reads V^T K-major instead of V MN-major.
    constexpr uint32_t kIdS = idesc_f16(FP8 ? false : BF16, kTileM, kTileN, false);
    constexpr uint32_t kIdO = idesc_f16(FP8 ? false : BF16, kTileM, D, !FP8);
    // Descriptors are built once per operand; a K-step only moves the start
    // address field (address / 16, the low bits of the descriptor), which never
    // carries out for shared-memory addresses.
    const uint64_t dq0 = sdesc_sw128(smem_u32(tiles + C::kOffQ), 16, 1024);
    const uint64_t dkv0 = sdesc_sw128(smem_u32(tiles + C::kOffKV), 16, 1024);
    const uint64_t dv0 = FP8 ? sdesc_sw128(smem_u32(tiles + C::kOffKV), 16, 1024)
                             : sdesc_sw128(smem_u32(tiles + C::kOffKV), C::kBoxBytes, 1024);

    int acquired = 0;        // ring items acquired so far
    uint32_t pv_par = 0;     // bit t: parity of stream t's next p_full phase
    uint32_t q_par = 0;      // bit t: parity of stream t's next q_full phase
    bool ok = true;

    auto acquire = [&](int it) -> bool {
        if (acquired > it) return true;
        do {
            if (!__all_sync(0xffffffffu, wait_bar(&sh.kv_full[acquired % C::kStages], (acquired / C::kStages) & 1, abort_flag)))
                return false;
        } while (++acquired <= it);
        tc_fence_after();
        return true;
    };
    auto issue_s = [&](int t, int item, bool release) {
        const uint64_t da = dq0 + ((t * C::kTileBytes) >> 4);
        const uint64_t db = dkv0 + (((item % C::kStages) * C::kTileBytes) >> 4);
        const uint32_t d = tmem + C::tm_s(t);
        // K-step kk reads 32 bytes of each 128-byte row of Q and K (16 16-bit or 32
        // 8-bit elements of D), in box kk / 4
        if constexpr (FP8) {
            umma_ss_x4<true, StepOffsets<StepsK4, StepsK4>>(d, da, db, kIdS, 0);
        } else if constexpr (D == 128) {
            using K8 = StepsK8<(C::kBoxBytes >> 4)>;
            umma_ss_x8<StepOffsets<K8, K8>>(d, da, db, kIdS, 0);
        } else {
            umma_ss_x4<false, StepOffsets<StepsK4, StepsK4>>(d, da, db, kIdS, 0);
        }
        umma_commit_elect(&sh.s_full[t]);
        if (release) umma_commit_elect(&sh.kv_empty[item % C::kStages]);
    };
    auto issue_pv = [&](int t, int item, bool first, bool release) {
        const uint64_t dv = dv0 + (((item % C::kStages) * C::kTileBytes) >> 4);
        const uint32_t d = tmem + C::tm_o(t), a = tmem + C::tm_s(t);
        if constexpr (FP8) {
            // K-step kk reads 32 keys: 8 TMEM columns of E4M3 P, 32 bytes of each V^T row
            umma_ts_x4_f8<StepOffsets<StepsCol4, StepsK4>>(d, a, dv, kIdO, first ? 0u : 1u);
        } else {
            // K-step kk reads 16 keys = 2048 bytes of V and 8 TMEM columns of P
            umma_ts_x8<StepOffsets<StepsCol8, StepsMN8>>(d, a, dv, kIdO, first ? 0u : 1u);
        }
        umma_commit_elect(&sh.pv_done[t]);
        if (release) umma_commit_elect(&sh.kv_empty[item % C::kStages]);
    };
    // First S of stream t in work tile w (ring items from `base`); it releases
    // K_0 unless the other stream reads it and has not issued its first S yet.
    // (Key split: each stream reads its own K/V tiles, ring items 2 (2 j + t) and
    // 2 (2 j + t) + 1 of a work tile, each read once.)
    auto start_stream = [&](int t, const Tile& w, int base, bool other_done) -> bool {
        if (!__all_sync(0xffffffffu, wait_bar(&sh.q_full[t], (q_par >> t) & 1, abort_flag))) return false;
        q_par ^= 1u << t;
        const int item = KS ? base + 2 * t : base;
        if (!acquire(item)) return false;
        issue_s(t, item, KS || w.nkv[kNumQ - 1 - t] == 0 || other_done);
        if (w.nkv[t] == 1) umma_commit_elect(&sh.q_empty[t]);   // that was its last S of this work tile
        return true;
    };

    int k = 0;
    int idx = tile_index(0, p.n_tiles);
    if (idx < 0) return;
    Tile cur = make_tile<CAUSAL, SPLIT, KS>(p, idx);
    int cur_base = 0;
    uint32_t started = 0;    // bit t: first S of `cur` already issued by the previous tile
    while (ok) {
        const int nidx = tile_index(k + 1, p.n_tiles);
        const bool has_next = nidx >= 0;
        const Tile nxt = has_next ? make_tile<CAUSAL, SPLIT, KS>(p, nidx) : cur;
        const int nxt_base = cur_base + (KS ? 2 * (cur.nkv[0] + cur.nkv[1]) : 2 * cur.n_all);
        if (ok && cur.nkv[0] > 0 && !(started & 1u)) {
            ok = start_stream(0, cur, cur_base, (started & 2u) != 0);
            started |= 1u;
        }
        if (ok && cur.nkv[1] > 0 && !(started & 2u)) ok = start_stream(1, cur, cur_base, true);
        uint32_t nstarted = 0;
        for (int j = 0; j < cur.n_all && ok; ++j) {
#pragma unroll
            for (int t = 0; t < kNumQ; ++t) {
                if (!ok || j >= cur.nkv[t]) continue;
                const int item_v = KS ? cur_base + 2 * (2 * j + t) + 1 : cur_base + 2 * j + 1;
                const bool more = j + 1 < cur.nkv[t];
                // V_j, K_{j+1} (long since landed) and P_t: the three barriers
                // are tested together so their latencies overlap; only a test
                // that fails falls back to a bounded wait.
                const int next_k = KS ? cur_base + 2 * (2 * (j + 1) + t) : item_v + 1;
                const int need = more ? next_k : item_v;
                const int item_k = more ? next_k : item_v;
                const uint32_t got = mbar_test3_bcast(&sh.kv_full[item_v % C::kStages], (item_v / C::kStages) & 1,
                                                      &sh.kv_full[item_k % C::kStages], (item_k / C::kStages) & 1,
                                                      &sh.p_full[t], (pv_par >> t) & 1);
                const bool r_p = (got & 4u) != 0;
                if ((got & 3u) == 3u && acquired >= item_v && acquired <= need) {
                    acquired = need + 1;   // both tested complete above
                    tc_fence_after();
                }
                if (!acquire(need) ||
                    (!r_p && !__all_sync(0xffffffffu, wait_bar(&sh.p_full[t], (pv_par >> t) & 1, abort_flag)))) {
                    ok = false;
                    continue;
                }
                tc_fence_after();
                pv_par ^= 1u << t;
                issue_pv(t, item_v, j == 0, KS || t == kNumQ - 1 || j >= cur.nkv[kNumQ - 1]);
                if (more) {
                    issue_s(t, next_k, KS || t == kNumQ - 1 || j + 1 >= cur.nkv[kNumQ - 1]);
                    if (j + 2 == cur.nkv[t]) umma_commit_elect(&sh.q_empty[t]);
                } else if (has_next && nxt.nkv[t] > 0) {
                    ok = start_stream(t, nxt, nxt_base, ((nstarted >> (kNumQ - 1 - t)) & 1u) != 0);
                    nstarted |= 1u << t;
                }
            }
        }
        if (!ok || !has_next) break;
        ++k;
        cur = nxt;
        cur_base = nxt_base;
        started = nstarted;
    }
    if (!ok && lane_id() == 0) give_up(sh, ST_MMA);
    // Nothing of ours may still be in flight when the CTA retires.
    umma_commit_elect(&sh.drain);
    volatile int never = 0;
    if (!__all_sync(0xffffffffu, wait_bar(&sh.drain, 0, &never)) && lane_id() == 0) atomicOr(&g_fa_status, ST_DRAIN);
}

// FP8: the exponent coefficient of K/V tile jg (the Q scale times its K block
// scale), the log2 shift that folds its V block scale into P (relative to the
// head's largest, v_ref, times 2^kFp8Shift) and that shift's inverse factor.
// fold is 2^-shift up to the rounding of the approximate log2 and reciprocal;
// the row sums are multiplied by fold and O by v_ref / 2^kFp8Shift, so O stays
// a convex combination of the dequantized V rows with the weights actually used.
__device__ __forceinline__ void fp8_tile_scales(const Params& p, int kvh, int jg, float c_q, float v_ref,
                                                float lg_vref, float& c_s, float& shift, float& fold) {
    const size_t kb = static_cast<size_t>(kvh) * p.n_blocks + jg;
    const float vs = __ldg(p.v_scale + kb);
    c_s = c_q * __ldg(p.k_scale + kb);
    shift = kFp8Shift + (lg2_approx(vs) - lg_vref);
    fold = v_ref * rcp_approx(vs) * (1.f / kFp8ShiftScale);
}

template <int D, bool BF16, bool CAUSAL, bool SPLIT, bool FP8, bool KS>
__device__ void run_softmax(SharedState& sh, uint32_t tmem, int t, const Params& p) {
    static_assert(!(FP8 && SPLIT), "the FP8 path has no split-K form");
    static_assert(!(KS && (FP8 || SPLIT)), "the key split is a 16-bit, single-pass form");
    constexpr float kLazy = FP8 ? kLazyRescaleFp8 : kLazyRescale;
    volatile int* abort_flag = &sh.abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = threadIdx.x - 128 * (1 + t);               // row of this thread in Q tile t
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t ts = tmem + lane_addr + Cfg<D>::tm_s(t);
    const uint32_t to = tmem + lane_addr + Cfg<D>::tm_o(t);
    const float scale_log2 = p.scale_log2;
    const int N = p.N;
    int step = 0;   // S/P steps of this stream so far (phase of s_full / p_full / alpha_ready / pv_done)
    int kph = 0;    // key split: exchanges with the other stream so far (phase of k_sync)
    bool ok = true;

    for (int k = 0; ok; ++k) {
        const int idx = tile_index(k, p.n_tiles);
        if (idx < 0) break;
        const Tile w = make_tile<CAUSAL, SPLIT, KS>(p, idx);
        const int nkv_t = w.nkv[t];
        const int qi = stream_row0<KS>(w, t) + r;             // row of this thread in its Q plane
        const size_t row_g = static_cast<size_t>(w.bh) * N + qi;
        if (!KS && nkv_t == 0) {
            // split mode: this chunk holds none of the stream's keys
            if (SPLIT && qi < N)
                p.ws_st[static_cast<size_t>(w.split) * p.BH * N + row_g] = make_float4(-INFINITY, 0.f, 0.f, 0.f);
            continue;
        }

        // FP8: S is the product of the E4M3 values; the scores are S times the
        // Q and K block scales, folded into the exponent's coefficient.  P V adds
        // E4M3 V^T bytes: each tile's V block scale, relative to the head's largest
        // (v_ref), and a range shift of 2^kFp8Shift are folded into P (see the pack below).
        float c_q = scale_log2, v_ref = 1.f;
        if constexpr (FP8) {
            c_q = scale_log2 * __ldg(p.q_scale + static_cast<size_t>(w.bh) * p.n_blocks + (w.q0 + kTileM * t) / kTileM);
            float vm = 0.f;
            for (int b = lane; b < p.n_blocks; b += 32)
                vm = fmaxf(vm, __ldg(p.v_scale + static_cast<size_t>(w.kvh) * p.n_blocks + b));
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, m));
            v_ref = vm;
        }
        float m_ref = -INFINITY;   // reference max, log2 units of the scaled score
        float l = 0.f;             // running sum that normalises O (see the row sums below)
        float ls = 0.f;            // running sum of the unrounded p, for the log-sum-exp
        // Coefficient, P shift (log2) and 2^-shift of the next step.  FP8 loads
        // the next K/V tile's scales one step ahead, off the step's critical path.
        float c_nx = scale_log2, sh_nx = 0.f, fo_nx = 1.f, lg_vref = 0.f;
        if constexpr (FP8) {
            lg_vref = lg2_approx(v_ref);
            fp8_tile_scales(p, w.kvh, SPLIT ? w.j0 : 0, c_q, v_ref, lg_vref, c_nx, sh_nx, fo_nx);
        }
        for (int j = 0; j < nkv_t; ++j, ++step) {
            ok = __all_sync(0xffffffffu, wait_bar(&sh.s_full[t], step & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            float s[kTileN];
            tmem_ld128_wait(ts, s);

            const int jg = (SPLIT || KS) ? stream_kv0<KS>(w, t) + j : j;   // global K/V tile index
            const int k0 = jg * kTileN;
            const float c_s = c_nx, shift = sh_nx, fold = fo_nx;
            // Causal: the row's query is the token at position qpos of the key
            // sequence (qi + Nk - Nq; with stacked heads, its position within its
            // head).  A tile needs the element mask if it holds a key past the
            // smallest position of the stream's rows, or keys past Nk.  (Read from
            // the kernel parameters here, not kept live across the loop.)
            const bool need_mask = (CAUSAL && k0 + kTileN - 1 > (p.packed ? 0 : stream_row0<KS>(w, t)) + p.causal_off) ||
                                   (k0 + kTileN > p.Nk);
            if (need_mask) {
                const int qpos = (p.packed ? qi % p.q_per : qi) + p.causal_off;
                const int Nk = p.Nk;
#pragma unroll
                for (int c = 0; c < kTileN; ++c) {
                    const int key = k0 + c;
                    if (key >= Nk || (CAUSAL && key > qpos)) s[c] = -INFINITY;
                }
            }
            // Row max of the raw scores (three-input max), then into log2 units.
            float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
            for (int c = 4; c < kTileN; c += 8) {
                mx[0] = fmax3(mx[0], s[c], s[c + 1]);
                mx[1] = fmax3(mx[1], s[c + 2], s[c + 3]);
                if (c + 4 < kTileN) {
                    mx[2] = fmax3(mx[2], s[c + 4], s[c + 5]);
                    mx[3] = fmax3(mx[3], s[c + 6], s[c + 7]);
                }
            }
            const float m_tile = fmax3(fmaxf(mx[0], mx[1]), mx[2], mx[3]) * c_s;
            const float m_new = fmaxf(m_ref, m_tile);
            float alpha = 1.f;
            if (m_ref == -INFINITY) {
                alpha = 0.f;            // nothing accumulated yet
                m_ref = m_new;
            } else if (m_new > m_ref + kLazy) {
                alpha = ex2_approx(m_ref - m_new);
                m_ref = m_new;
            }
            sh.alpha[t][r] = alpha;
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.alpha_ready[t]);

            // p = 2^(s*c - m_ref), one rounding of the fused product-difference.
            // m_ref = round(max * c) is the same reference for every element of
            // the row, so it need not equal the exact max: the row's largest
            // element gets an exponent within half an ulp of m_ref of zero.  For
            // |m_ref| >= 2^24 that half ulp is more than a unit and could
            // overflow 16-bit P, so such rows round the product on its own and
            // subtract after (then the largest element maps to exactly 2^0).
            const float msub = (m_ref == -INFINITY) ? 0.f : m_ref;
            const bool fused = fabsf(msub) < 16777216.f;
            if (!fused) {
                // The product is rounded on its own first and the loop below only
                // subtracts (coefficient 1).  One loop body serves both cases: a
                // second unrolled copy of it costs instruction-cache misses.
#pragma unroll
                for (int c = 0; c < kTileN; ++c) s[c] = __fmul_rn(s[c], c_s);
            }
            const float cf = fused ? c_s : 1.f;
            const uint64_t c2 = pack_f32x2(cf, cf);
            const uint64_t nm2 = pack_f32x2(shift - msub, shift - msub);
            if constexpr (FP8) {
                // P'' = 2^(s c - m_ref + shift) = p * 2^kFp8Shift * vs / v_ref, four per E4M3 word
                uint64_t lx2 = pack_f32x2(0.f, 0.f);   // sum of the unrounded P''
                uint32_t pk8[kTileN / 4];
#pragma unroll
                for (int i = 0; i < kTileN / 4; ++i) {
                    float x0, x1, x2, x3;
                    unpack_f32x2(fma_f32x2(pack_f32x2(s[4 * i], s[4 * i + 1]), c2, nm2), x0, x1);
                    unpack_f32x2(fma_f32x2(pack_f32x2(s[4 * i + 2], s[4 * i + 3]), c2, nm2), x2, x3);
                    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(x2), p3 = ex2_approx(x3);
                    pk8[i] = pack_e4m3x4(p0, p1, p2, p3);
                    lx2 = add_f32x2(lx2, add_f32x2(pack_f32x2(p0, p1), pack_f32x2(p2, p3)));
                }
                tmem_st32(ts, pk8);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.p_full[t]);
                if (j + 1 < nkv_t) fp8_tile_scales(p, w.kvh, jg + 1, c_q, v_ref, lg_vref, c_nx, sh_nx, fo_nx);
                // Row sums of the E4M3 P actually used by P V (normalises O), and of
                // the unrounded P'' (the log-sum-exp), both back in units of p.
                float lr[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < kTileN / 4; ++i) add_e4m3x4(pk8[i], lr[2 * (i & 1)], lr[2 * (i & 1) + 1]);
                float x0, x1;
                unpack_f32x2(lx2, x0, x1);
                l = l * alpha + ((lr[0] + lr[1]) + (lr[2] + lr[3])) * fold;
                ls = ls * alpha + (x0 + x1) * fold;
            } else {
            uint64_t lx2 = pack_f32x2(0.f, 0.f);   // sum of the fp32 p
            uint32_t pk[kTileN / 2];                 // P as packed 16-bit pairs
#pragma unroll
            for (int i = 0; i < kTileN / 2; ++i) {
                float x0, x1;
                unpack_f32x2(fma_f32x2(pack_f32x2(s[2 * i], s[2 * i + 1]), c2, nm2), x0, x1);
                const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                if constexpr (BF16) {
                    pk[i] = pack_bf16x2(p0, p1);
                    lx2 = add_f32x2(lx2, pack_f32x2(p0, p1));
                } else {
                    pk[i] = pack_f16x2(p0, p1);
                    lx2 = add_f32x2(lx2, pack_f32x2(p0, p1));
                }
            }
            tmem_st32(ts, reinterpret_cast<const uint32_t(&)[32]>(pk[0]));
            tmem_st32(ts + 32, reinterpret_cast<const uint32_t(&)[32]>(pk[32]));
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.p_full[t]);

            // The row sums are not needed by the tensor core: they run while it
            // does this stream's P V and next S.  bf16 normalises O by the sum of
            // the rounded P that P V actually used (a lone p near 1 rounded to bf16
            // is off by up to 2^-8, which would bias O by as much); fp16 P is
            // within 2^-11 of p, so fp16 normalises by the sum of the fp32 p, the
            // pages' own l, already accumulated in the exponent loop.
            if constexpr (BF16) {
                float lr[4] = {0.f, 0.f, 0.f, 0.f};     // sums of the rounded bf16 P
#pragma unroll
                for (int i = 0; i < kTileN / 2; ++i) {
                    lr[i & 3] = add_lo_bf16(pk[i], lr[i & 3]);
                    lr[(i + 2) & 3] = add_hi_bf16(pk[i], lr[(i + 2) & 3]);
                }
                l = l * alpha + ((lr[0] + lr[1]) + (lr[2] + lr[3]));
                float x0, x1;
                unpack_f32x2(lx2, x0, x1);
                ls = ls * alpha + (x0 + x1);
            } else {
                float x0, x1;
                unpack_f32x2(lx2, x0, x1);
                l = l * alpha + (x0 + x1);
                ls = l;
            }
            }   // 16-bit P
        }
        if (!ok) break;

        if constexpr (KS) {
            // Key split: merge the two streams' partials of these rows.  Each
            // stream publishes (m_ref, l, ls) once its last P V is complete; then
            // each combines its half of the O columns from both O_0 and O_1:
            //   m = max(m_0, m_1), a_s = 2^(m_s - m), O = sum_s a_s O_s / sum_s a_s l_s.
            const int quarter = warp & 3;
            auto exchange = [&]() -> bool {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.k_sync[quarter]);
                const bool got = __all_sync(0xffffffffu, wait_bar(&sh.k_sync[quarter], kph & 1, abort_flag));
                ++kph;
                tc_fence_after();
                return got;
            };
            if (nkv_t > 0) {
                ok = __all_sync(0xffffffffu, wait_bar(&sh.pv_done[t], (step - 1) & 1, abort_flag));
                if (!ok) break;
            }
            sh.k_part[t][r] = make_float4(m_ref, l, ls, 0.f);
            if (!exchange()) {
                ok = false;
                break;
            }
            const float4 other = sh.k_part[t ^ 1][r];
            const float mm = fmaxf(m_ref, other.x);
            const float a_me = m_ref == -INFINITY ? 0.f : ex2_approx(m_ref - mm);
            const float a_ot = other.x == -INFINITY ? 0.f : ex2_approx(other.x - mm);
            const float lt = a_me * l + a_ot * other.y, lst = a_me * ls + a_ot * other.z;
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
            const bool row_ok = qi < N;
            constexpr int kHalf = D / 2;   // O columns this stream writes
            const uint32_t o_me = tmem + lane_addr + Cfg<D>::tm_o(t) + kHalf * t;
            const uint32_t o_ot = tmem + lane_addr + Cfg<D>::tm_o(t ^ 1) + kHalf * t;
            uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + (row_ok ? row_g : 0) * D + kHalf * t);
#pragma unroll
            for (int c = 0; c < kHalf; c += 32) {
                uint32_t va[32], vb[32];
                tmem_ld32_wait(o_me + c, va);
                tmem_ld32_wait(o_ot + c, vb);
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float x[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        // a stream without keys left its O unwritten: its term is 0, not 0 * O
                        const float pa = a_me != 0.f ? a_me * __uint_as_float(va[2 * i + h]) : 0.f;
                        const float pb = a_ot != 0.f ? a_ot * __uint_as_float(vb[2 * i + h]) : 0.f;
                        x[h] = (pa + pb) * inv;
                    }
                    pk[i] = BF16 ? pack_bf16x2(x[0], x[1]) : pack_f16x2(x[0], x[1]);
                }
                if (row_ok) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        orow[c / 8 + q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                }
            }
            if (row_ok && t == 0) p.lse[row_g] = lst > 0.f ? (mm + log2f(lst)) * 0.69314718055994531f : -INFINITY;
            // Both streams have read O_0 and O_1 before either's next P V overwrites them.
            if (!exchange()) {
                ok = false;
                break;
            }
            tc_fence_before();
            continue;
        }

        // Epilogue of this work tile: wait for the last P V, then O / l -> 16-bit
        // -> global (rows past N are not written) and the LSE.
        ok = __all_sync(0xffffffffu, wait_bar(&sh.pv_done[t], (step - 1) & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        const bool row_ok = qi < N;
        if constexpr (SPLIT) {
            // split mode: the unnormalised partial and its (m, l) go to the workspace
            const size_t prow = static_cast<size_t>(w.split) * p.BH * N + row_g;
            float4* dst = reinterpret_cast<float4*>(p.ws_o + prow * D);
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                uint32_t v[32];
                tmem_ld32_wait(to + c, v);
                if (row_ok) {
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        dst[c / 4 + q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                                     __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
                }
            }
            if (row_ok) p.ws_st[prow] = make_float4(m_ref, l, ls, 0.f);
            tc_fence_before();
            continue;
        }
        // FP8: O holds sum P'' v8 = 2^kFp8Shift / v_ref * sum p (vs v8); undo the fold
        const float inv = l > 0.f ? (FP8 ? v_ref / kFp8ShiftScale : 1.f) / l : 0.f;
        uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + (row_ok ? row_g : 0) * D);
#pragma unroll
        for (int c = 0; c < D; c += 32) {
            uint32_t v[32];
            tmem_ld32_wait(to + c, v);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float x0 = __uint_as_float(v[2 * i]) * inv, x1 = __uint_as_float(v[2 * i + 1]) * inv;
                pk[i] = BF16 ? pack_bf16x2(x0, x1) : pack_f16x2(x0, x1);
            }
            if (row_ok) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    orow[c / 8 + q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
        }
        if (row_ok)
            p.lse[row_g] =
                ls > 0.f ? (m_ref + log2f(ls)) * 0.69314718055994531f : -INFINITY;
        // The next work tile's first P V overwrites O_t; it waits for this
        // stream's next p_full, which comes after these loads.
        tc_fence_before();
    }
    if (!ok) give_up(sh, ST_SOFTMAX);
}

template <int D, bool CAUSAL, bool SPLIT, bool KS>
__device__ void run_correction(SharedState& sh, uint32_t tmem, const Params& p) {
    using C = Cfg<D>;
    volatile int* abort_flag = &sh.abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = threadIdx.x - 128 * (1 + kNumQ);
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    int steps[kNumQ] = {0, 0};
    bool ok = true;
    for (int k = 0; ok; ++k) {
        const int idx = tile_index(k, p.n_tiles);
        if (idx < 0) break;
        const Tile w = make_tile<CAUSAL, SPLIT, KS>(p, idx);
        for (int j = 0; j < w.n_all && ok; ++j) {
            for (int t = 0; t < kNumQ; ++t) {
                if (j >= w.nkv[t]) continue;
                ok = __all_sync(0xffffffffu, wait_bar(&sh.alpha_ready[t], steps[t] & 1, abort_flag));
                if (!ok) break;
                if (j > 0) {
                    const float a = sh.alpha[t][r];
                    if (__any_sync(0xffffffffu, a != 1.f)) {
                        // O_t holds P V of steps < j; the last of them finished before S_t(j) did.
                        ok = __all_sync(0xffffffffu, wait_bar(&sh.pv_done[t], (steps[t] - 1) & 1, abort_flag));
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t to = tmem + lane_addr + C::tm_o(t);
#pragma unroll
                        for (int c = 0; c < D; c += 32) {
                            uint32_t v[32];
                            tmem_ld32_wait(to + c, v);
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * a);
                            tmem_st32(to + c, v);
                        }
                        tmem_st_wait();
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.p_full[t]);
                ++steps[t];
            }
        }
    }
    if (!ok) give_up(sh, ST_CORRECTION);
}

template <int D, bool BF16, bool CAUSAL, bool SPLIT, bool FP8 = false, bool KS = false>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const Params p) {
    using C = Cfg<D, FP8>;
    extern __shared__ uint8_t dyn_smem[];
    __shared__ SharedState sh;
    uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, wg = warp >> 2;

    if (threadIdx.x == 0) {
        for (int t = 0; t < kNumQ; ++t) {
            mbar_init(&sh.q_full[t], 1);
            mbar_init(&sh.q_empty[t], 1);
            mbar_init(&sh.s_full[t], 1);
            mbar_init(&sh.p_full[t], 8);   // 4 softmax warps + 4 correction warps
            mbar_init(&sh.alpha_ready[t], 4);
            mbar_init(&sh.pv_done[t], 1);
        }
        for (int q = 0; q < 4; ++q) mbar_init(&sh.k_sync[q], kNumQ);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&sh.kv_full[s], 1);
            mbar_init(&sh.kv_empty[s], 1);
        }
        mbar_init(&sh.drain, 1);
        sh.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&sh.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    if (wg == 0) {
        setmaxnreg_dec<96>();
        if (warp == 0 && lane == 0)
            run_kv_producer<D, CAUSAL, SPLIT, FP8, KS>(sh, tiles, &tm_k, &tm_v, p);
        else if (warp == 1)
            run_mma<D, BF16, CAUSAL, SPLIT, FP8, KS>(sh, tiles, tmem, p);
        else if (warp == 2 && lane == 0)
            run_q_producer<D, CAUSAL, SPLIT, FP8, KS>(sh, tiles, &tm_q, p);
        __syncwarp();
    } else if (wg <= kNumQ) {
        setmaxnreg_inc<176>();
        run_softmax<D, BF16, CAUSAL, SPLIT, FP8, KS>(sh, tmem, wg - 1, p);
    } else {
        setmaxnreg_dec<64>();
        run_correction<D, CAUSAL, SPLIT, KS>(sh, tmem, p);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Merge of the split partials, one warp per query row (HBM-bound):
//   m = max_s m_s,  w_s = 2^(m_s - m),  O = sum_s w_s O_s / sum_s w_s l_s,
//   LSE = (m + log2 sum_s w_s l_exact_s) * ln 2,
// skipping partials with l_s = 0 (chunks without a visible key).
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_merge_kernel(const float* __restrict__ ws_o,
                                                       const float4* __restrict__ ws_st, void* o, float* lse,
                                                       long long rows, int n_splits) {
    constexpr int kPer = D / 32;   // elements of the row per lane
    const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float m = -INFINITY;
    for (int s = 0; s < n_splits; ++s) {
        const float4 st = ws_st[static_cast<size_t>(s) * rows + row];
        if (st.y > 0.f) m = fmaxf(m, st.x);
    }
    float wsum = 0.f, lsum = 0.f, acc[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
    for (int s = 0; s < n_splits; ++s) {
        const float4 st = ws_st[static_cast<size_t>(s) * rows + row];
        if (!(st.y > 0.f)) continue;
        const float wgt = exp2f(st.x - m);
        wsum += wgt * st.y;
        lsum += wgt * st.z;
        const float* src = ws_o + (static_cast<size_t>(s) * rows + row) * D + lane * kPer;
        if constexpr (kPer == 4) {
            const float4 x = *reinterpret_cast<const float4*>(src);
            acc[0] += wgt * x.x; acc[1] += wgt * x.y; acc[2] += wgt * x.z; acc[3] += wgt * x.w;
        } else {
            const float2 x = *reinterpret_cast<const float2*>(src);
            acc[0] += wgt * x.x; acc[1] += wgt * x.y;
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    uint32_t pk[kPer / 2];
#pragma unroll
    for (int i = 0; i < kPer / 2; ++i)
        pk[i] = BF16 ? pack_bf16x2(acc[2 * i] * inv, acc[2 * i + 1] * inv) : pack_f16x2(acc[2 * i] * inv, acc[2 * i + 1] * inv);
    uint16_t* orow = static_cast<uint16_t*>(o) + static_cast<size_t>(row) * D + lane * kPer;
    if constexpr (kPer == 4)
        *reinterpret_cast<uint2*>(orow) = make_uint2(pk[0], pk[1]);
    else
        *reinterpret_cast<uint32_t*>(orow) = pk[0];
    if (lane == 0) lse[row] = lsum > 0.f ? (m + log2f(lsum)) * 0.69314718055994531f : -INFINITY;
}

// One warp waits, with the forward kernel's own bounded wait, on an mbarrier
// that nothing arrives on: the wait gives up after its time limit, records a
// status bit and the kernel returns normally.
__global__ void __launch_bounds__(32) selftest_wait_timeout_kernel() {
    __shared__ SharedState sh;
    if (threadIdx.x == 0) {
        mbar_init(&sh.drain, 1);
        sh.abort_flag = 0;
        fence_mbar_init();
    }
    __syncwarp();
    const bool ok = __all_sync(0xffffffffu, wait_bar(&sh.drain, 0, &sh.abort_flag));
    if (!ok && threadIdx.x == 0) give_up(sh, ST_SELFTEST);
}

// ------------------------------------------------------------------ host

template <int D, bool BF16, bool CAUSAL, bool SPLIT, bool FP8 = false, bool KS = false>
static cudaError_t launch(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const Params& p,
                          cudaStream_t stream) {
    auto kern = fa_fwd_kernel<D, BF16, CAUSAL, SPLIT, FP8, KS>;
    static std::atomic<uint64_t> configured{0};   // one bit per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (!bit || !(configured.load() & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D, FP8>::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    const int sms = sm_count(dev);
    if (sms <= 0) return cudaErrorInvalidDevice;
    const unsigned grid = static_cast<unsigned>(p.n_tiles < sms ? p.n_tiles : sms);
    kern<<<grid, kThreads, Cfg<D, FP8>::kSmemBytes, stream>>>(q, k, v, p);
    return cudaGetLastError();
}

}  // namespace fa103

using namespace fa103;

namespace fa103 {

// The argument checks of the 16-bit forward entry points, alone (no CUDA call
// is made): FA_OK or the status the entry point returns.
static int check_args(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv,
                      int Nq, int Nk, int D, float scale, int causal, int dtype, int n_splits, bool pack) {
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return FA_ERR_INVALID_ARG;
    if (H_kv < 1 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (causal && Nq > Nk) return FA_ERR_INVALID_ARG;
    if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    const void* ptrs[5] = {q, k, v, o, lse};
    for (const void* ptr : ptrs)
        if (ptr == nullptr || (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0) return FA_ERR_MISALIGNED;
    const uint64_t BH = static_cast<uint64_t>(B) * static_cast<uint64_t>(H);
    const uint64_t BHkv = static_cast<uint64_t>(B) * static_cast<uint64_t>(H_kv);
    const uint64_t q_elems = BH * static_cast<uint64_t>(Nq) * static_cast<uint64_t>(D);
    const uint64_t kv_elems = BHkv * static_cast<uint64_t>(Nk) * static_cast<uint64_t>(D);
    if (BH > 0x7fffffffull || q_elems >= (uint64_t(1) << 40) || kv_elems >= (uint64_t(1) << 40))
        return FA_ERR_INVALID_ARG;
    const uint64_t planes = pack ? BHkv : BH;
    const uint64_t rows = pack ? static_cast<uint64_t>(H / H_kv) * Nq : static_cast<uint64_t>(Nq);
    if (rows > 0x7fffffffull) return FA_ERR_INVALID_ARG;
    const uint64_t n_qblocks = (rows + kRowsPerTile - 1) / kRowsPerTile;
    if (n_qblocks * planes * static_cast<uint64_t>(n_splits) > 0x7fffffffull) return FA_ERR_INVALID_ARG;
    const size_t tbytes = static_cast<size_t>(q_elems) * 2, lbytes = static_cast<size_t>(BH) * Nq * sizeof(float);
    const size_t kvbytes = static_cast<size_t>(kv_elems) * 2;
    const void* ins[3] = {q, k, v};
    const size_t in_bytes[3] = {tbytes, kvbytes, kvbytes};
    for (int i = 0; i < 3; ++i)
        if (overlaps(o, tbytes, ins[i], in_bytes[i]) || overlaps(lse, lbytes, ins[i], in_bytes[i]))
            return FA_ERR_INVALID_ARG;
    if (overlaps(o, tbytes, lse, lbytes)) return FA_ERR_INVALID_ARG;
    return FA_OK;
}

// Argument checks and kernel parameters shared by the 16-bit forward entry
// points.  Q, O, LSE have Nq rows per head, K and V Nk rows per K/V head.  With
// `pack`, the query heads that share a K/V head are stacked into one Q plane of
// (H / H_kv) * Nq rows (their rows are adjacent in memory), so one K/V head is
// streamed once for all of them.
static int prepare(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int Nq,
                   int Nk, int D, float scale, int causal, int dtype, int n_splits, bool pack, CUtensorMap (&maps)[3],
                   Params& p) {
    const int st = check_args(q, k, v, o, lse, B, H, H_kv, Nq, Nk, D, scale, causal, dtype, n_splits, pack);
    if (st != FA_OK) return st;
    const uint64_t BH = static_cast<uint64_t>(B) * static_cast<uint64_t>(H);
    const uint64_t BHkv = static_cast<uint64_t>(B) * static_cast<uint64_t>(H_kv);
    const uint64_t planes = pack ? BHkv : BH;
    const uint64_t rows = pack ? static_cast<uint64_t>(H / H_kv) * Nq : static_cast<uint64_t>(Nq);
    const uint64_t n_qblocks = (rows + kRowsPerTile - 1) / kRowsPerTile;
    if (!make_tile_map(&maps[0], q, dtype, D, static_cast<int>(rows), static_cast<int>(planes)) ||
        !make_tile_map(&maps[1], k, dtype, D, Nk, static_cast<int>(BHkv)) ||
        !make_tile_map(&maps[2], v, dtype, D, Nk, static_cast<int>(BHkv)))
        return FA_ERR_CUDA;
    p.o = o;
    p.lse = lse;
    p.ws_o = nullptr;
    p.ws_st = nullptr;
    p.N = static_cast<int>(rows);
    p.Nk = Nk;
    p.q_per = Nq;
    p.causal_off = Nk - Nq;
    p.packed = pack ? 1 : 0;
    p.BH = static_cast<int>(planes);
    p.H = pack ? H_kv : H;
    p.kv_group = pack ? 1 : H / H_kv;
    p.n_qblocks = static_cast<int>(n_qblocks);
    p.n_splits = n_splits;
    p.n_tiles = static_cast<int>(n_qblocks * planes * static_cast<uint64_t>(n_splits));
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.q_scale = p.k_scale = p.v_scale = nullptr;
    p.n_blocks = 0;
    p.fault_item = -1;
    return FA_OK;
}

template <bool SPLIT, bool KS>
static int dispatch_as(const CUtensorMap (&m)[3], const Params& p, int D, int dtype, int causal,
                       cudaStream_t stream) {
    cudaError_t e;
    const bool bf = dtype == FA_BF16;
#define FA_LAUNCH(DD, BB, CC) e = launch<DD, BB, CC, SPLIT, false, KS>(m[0], m[1], m[2], p, stream)
    if (D == 64) {
        if (bf) { if (causal) FA_LAUNCH(64, true, true); else FA_LAUNCH(64, true, false); }
        else    { if (causal) FA_LAUNCH(64, false, true); else FA_LAUNCH(64, false, false); }
    } else {
        if (bf) { if (causal) FA_LAUNCH(128, true, true); else FA_LAUNCH(128, true, false); }
        else    { if (causal) FA_LAUNCH(128, false, true); else FA_LAUNCH(128, false, false); }
    }
#undef FA_LAUNCH
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// The 16-bit forward launch.  With no more 256-row work tiles than SMs (short
// sequences, few heads), a CTA would run one tile's chains back to back with
// SMs left idle; the key split then deals 128-row Q tiles instead, each with
// its K/V tiles shared out between the CTA's two streams (half the chain) and
// merged on chip.  The choice is made on `ks_tiles` 256-row work tiles (< 0:
// this launch's).
template <bool SPLIT>
static int dispatch(const CUtensorMap (&m)[3], const Params& p, int D, int dtype, int causal, cudaStream_t stream,
                    long long ks_tiles = -1) {
    if constexpr (!SPLIT) {
        if (!p.packed) {
            int dev = 0;
            if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
            const int sms = sm_count(dev);
            const long long tiles = ks_tiles < 0 ? p.n_tiles : ks_tiles;
            if (sms > 0 && tiles <= sms) {
                Params pk = p;
                pk.n_qblocks = (p.N + kTileM - 1) / kTileM;
                pk.n_tiles = pk.n_qblocks * p.BH;
                return dispatch_as<false, true>(m, pk, D, dtype, causal, stream);
            }
        }
    }
    return dispatch_as<SPLIT, false>(m, p, D, dtype, causal, stream);
}

static int dispatch_merge(const Params& p, int D, int dtype, cudaStream_t stream) {
    const long long rows = static_cast<long long>(p.BH) * p.N;
    const unsigned grid = static_cast<unsigned>((rows + 7) / 8);
    const bool bf = dtype == FA_BF16;
    if (D == 64) {
        if (bf) fa_merge_kernel<64, true><<<grid, 256, 0, stream>>>(p.ws_o, p.ws_st, p.o, p.lse, rows, p.n_splits);
        else    fa_merge_kernel<64, false><<<grid, 256, 0, stream>>>(p.ws_o, p.ws_st, p.o, p.lse, rows, p.n_splits);
    } else {
        if (bf) fa_merge_kernel<128, true><<<grid, 256, 0, stream>>>(p.ws_o, p.ws_st, p.o, p.lse, rows, p.n_splits);
        else    fa_merge_kernel<128, false><<<grid, 256, 0, stream>>>(p.ws_o, p.ws_st, p.o, p.lse, rows, p.n_splits);
    }
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

constexpr int kMaxSplits = 64;

static size_t splitkv_bytes(long long rows, int D, int n_splits) {
    return static_cast<size_t>(n_splits) * static_cast<size_t>(rows) * (static_cast<size_t>(D) * 4 + 16);
}

}  // namespace fa103

extern "C" int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int D,
                      float scale, int causal, int dtype, cudaStream_t stream) {
    CUtensorMap maps[3];
    Params p;
    const int st = prepare(q, k, v, o, lse, B, H, H, N, N, D, scale, causal, dtype, 1, false, maps, p);
    if (st != FA_OK) return st;
    return dispatch<false>(maps, p, D, dtype, causal, stream);
}

namespace fa103 {
// fa_fwd on planes [p0, p0 + H) of a B = 1 problem of `whole_planes` planes (the
// host-buffer pipeline's chunks): the key split is chosen for the whole
// problem, so the chunks' results equal fa_fwd's on the whole, bit for bit.
int fwd_part(const void* q, const void* k, const void* v, void* o, float* lse, int H, int N, int D, float scale,
             int causal, int dtype, long long whole_planes, cudaStream_t stream) {
    CUtensorMap maps[3];
    Params p;
    const int st = prepare(q, k, v, o, lse, 1, H, H, N, N, D, scale, causal, dtype, 1, false, maps, p);
    if (st != FA_OK) return st;
    return dispatch<false>(maps, p, D, dtype, causal, stream, static_cast<long long>(p.n_qblocks) * whole_planes);
}
}  // namespace fa103

extern "C" int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv,
                          int N, int D, float scale, int causal, int dtype, cudaStream_t stream) {
    CUtensorMap maps[3];
    Params p;
    const int st = prepare(q, k, v, o, lse, B, H, H_kv, N, N, D, scale, causal, dtype, 1, false, maps, p);
    if (st != FA_OK) return st;
    return dispatch<false>(maps, p, D, dtype, causal, stream);
}

extern "C" size_t fa_splitkv_workspace_bytes(int B, int H, int N, int D, int num_splits) {
    if (B < 1 || H < 1 || N < 1 || (D != 64 && D != 128) || num_splits < 1 || num_splits > kMaxSplits) return 0;
    return splitkv_bytes(static_cast<long long>(B) * H * N, D, num_splits);
}

extern "C" int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                              int N, int D, float scale, int causal, int dtype, int num_splits, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
    if (num_splits < 1 || num_splits > kMaxSplits) return FA_ERR_INVALID_ARG;
    const size_t need = fa_splitkv_workspace_bytes(B, H, N, D, num_splits);
    if (need != 0) {   // sizes valid: check the workspace before anything touches CUDA
        if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return FA_ERR_MISALIGNED;
        if (workspace_bytes < need) return FA_ERR_INVALID_ARG;
        const long long rows0 = static_cast<long long>(B) * H * N;
        const size_t tbytes = static_cast<size_t>(rows0) * D * 2, lbytes = static_cast<size_t>(rows0) * 4;
        const void* others[4] = {q, k, v, o};
        for (const void* x : others)
            if (x != nullptr && overlaps(workspace, need, x, tbytes)) return FA_ERR_INVALID_ARG;
        if (lse != nullptr && overlaps(workspace, need, lse, lbytes)) return FA_ERR_INVALID_ARG;
    }
    CUtensorMap maps[3];
    Params p;
    int st = prepare(q, k, v, o, lse, B, H, H, N, N, D, scale, causal, dtype, num_splits, false, maps, p);
    if (st != FA_OK) return st;
    const long long rows = static_cast<long long>(p.BH) * N;
    p.ws_o = static_cast<float*>(workspace);
    p.ws_st = reinterpret_cast<float4*>(static_cast<uint8_t*>(workspace) +
                                        static_cast<size_t>(num_splits) * rows * D * 4);
    st = dispatch<true>(maps, p, D, dtype, causal, stream);
    if (st != FA_OK) return st;
    return dispatch_merge(p, D, dtype, stream);
}

// ------------------------------------------------------------------ queries against a K/V sequence
extern "C" size_t fa_fwd_kv_workspace_bytes(int B, int H, int Nq, int D, int num_splits) {
    return fa_splitkv_workspace_bytes(B, H, Nq, D, num_splits);
}

extern "C" int fa_fwd_kv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv,
                         int Nq, int Nk, int D, float scale, int causal, int dtype, int num_splits, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
    if (num_splits < 0 || num_splits > kMaxSplits) return FA_ERR_INVALID_ARG;
    const int n_splits = num_splits > 0 ? num_splits : 1;
    if (num_splits > 0) {
        const size_t need = fa_fwd_kv_workspace_bytes(B, H, Nq, D, num_splits);
        if (need != 0) {   // sizes valid: check the workspace before anything touches CUDA
            if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return FA_ERR_MISALIGNED;
            if (workspace_bytes < need) return FA_ERR_INVALID_ARG;
            const size_t qb = static_cast<size_t>(B) * H * Nq * D * 2, lb = static_cast<size_t>(B) * H * Nq * 4;
            const size_t kvb = H_kv > 0 ? static_cast<size_t>(B) * H_kv * Nk * D * 2 : 0;
            const void* others[4] = {q, k, v, o};
            const size_t ob[4] = {qb, kvb, kvb, qb};
            for (int i = 0; i < 4; ++i)
                if (others[i] != nullptr && overlaps(workspace, need, others[i], ob[i])) return FA_ERR_INVALID_ARG;
            if (lse != nullptr && overlaps(workspace, need, lse, lb)) return FA_ERR_INVALID_ARG;
        }
    }
    // Few query rows per head (decode): stack the heads of a K/V group into one Q plane.
    const bool pack = H_kv > 0 && H % H_kv == 0 && H_kv < H && Nq < kTileM;
    CUtensorMap maps[3];
    Params p;
    int st = prepare(q, k, v, o, lse, B, H, H_kv, Nq, Nk, D, scale, causal, dtype, n_splits, pack, maps, p);
    if (st != FA_OK) return st;
    if (num_splits == 0) return dispatch<false>(maps, p, D, dtype, causal, stream);
    const long long rows = static_cast<long long>(p.BH) * p.N;
    p.ws_o = static_cast<float*>(workspace);
    p.ws_st = reinterpret_cast<float4*>(static_cast<uint8_t*>(workspace) +
                                        static_cast<size_t>(num_splits) * rows * D * 4);
    st = dispatch<true>(maps, p, D, dtype, causal, stream);
    if (st != FA_OK) return st;
    return dispatch_merge(p, D, dtype, stream);
}

// Split count for fa_fwd_kv: enough work tiles to cover the SMs once (twice
// for causal blocks of several query blocks, whose work per block differs),
// each chunk at least 4 K/V tiles, at most kMaxSplits; 0 when the unsplit grid
// already covers the SMs.
extern "C" int fa_fwd_kv_splits_hint(int B, int H, int H_kv, int Nq, int Nk, int D, int causal) {
    if (B < 1 || H < 1 || H_kv < 1 || Nq < 1 || Nk < 1 || H % H_kv != 0 || (D != 64 && D != 128)) return -1;
    if (causal != 0 && causal != 1) return -1;
    if (causal && Nq > Nk) return -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    const int sms = sm_count(dev);
    if (sms <= 0) return -1;
    const bool pack = H_kv < H && Nq < kTileM;
    const long long planes = static_cast<long long>(B) * (pack ? H_kv : H);
    const long long rows = pack ? static_cast<long long>(H / H_kv) * Nq : Nq;
    const long long qblocks = (rows + kRowsPerTile - 1) / kRowsPerTile;
    const long long base = planes * qblocks;
    const long long target = static_cast<long long>(sms) * ((causal && qblocks > 1) ? 2 : 1);
    if (base >= target) return 0;
    long long s = target / base;
    const long long kv_tiles = (static_cast<long long>(Nk) + kTileN - 1) / kTileN;
    if (s > kv_tiles / 4) s = kv_tiles / 4;
    if (s > kMaxSplits) s = kMaxSplits;
    return s >= 2 ? static_cast<int>(s) : 0;
}

// ------------------------------------------------------------------ FP8 forward
namespace fa103 {

// [BH, rows, inner] view of a contiguous byte tensor: 128-byte x 128-row boxes,
// 128-byte swizzle.  `inner` must make the row stride a multiple of 16 bytes.
static bool make_byte_map(CUtensorMap* map, const void* base, int inner, int rows, int BH) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows) * inner};
    cuuint32_t box[3] = {128, 128, 1};
    cuuint32_t elem_strides[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, elem_strides,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace fa103

extern "C" int fa_fwd_fp8(const void* q, const void* k, const void* v_t, const float* q_scale, const float* k_scale,
                          const float* v_scale, void* o, float* lse, int B, int H, int N, int D, float scale,
                          int causal, cudaStream_t stream) {
    if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    if (D != 128) return FA_ERR_UNSUPPORTED;
    if (N % 16 != 0) return FA_ERR_INVALID_ARG;   // V^T rows of N bytes: TMA strides are multiples of 16 bytes
    const void* ptrs[8] = {q, k, v_t, q_scale, k_scale, v_scale, o, lse};
    for (const void* ptr : ptrs)
        if (ptr == nullptr || (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0) return FA_ERR_MISALIGNED;
    const uint64_t BH = static_cast<uint64_t>(B) * static_cast<uint64_t>(H);
    const uint64_t elems = BH * static_cast<uint64_t>(N) * static_cast<uint64_t>(D);
    if (BH > 0x7fffffffull || elems >= (uint64_t(1) << 40)) return FA_ERR_INVALID_ARG;
    const uint64_t n_qblocks = (static_cast<uint64_t>(N) + kRowsPerTile - 1) / kRowsPerTile;
    if (n_qblocks * BH > 0x7fffffffull) return FA_ERR_INVALID_ARG;
    const int n_blocks = (N + kTileN - 1) / kTileN;
    const size_t in_bytes = static_cast<size_t>(elems), sc_bytes = static_cast<size_t>(BH) * n_blocks * 4;
    const size_t o_bytes = static_cast<size_t>(elems) * 2, l_bytes = static_cast<size_t>(BH) * N * 4;
    const void* ins[6] = {q, k, v_t, q_scale, k_scale, v_scale};
    const size_t ib[6] = {in_bytes, in_bytes, in_bytes, sc_bytes, sc_bytes, sc_bytes};
    for (int i = 0; i < 6; ++i)
        if (overlaps(o, o_bytes, ins[i], ib[i]) || overlaps(lse, l_bytes, ins[i], ib[i])) return FA_ERR_INVALID_ARG;
    if (overlaps(o, o_bytes, lse, l_bytes)) return FA_ERR_INVALID_ARG;
    CUtensorMap maps[3];
    const int bh = static_cast<int>(BH);
    if (!make_byte_map(&maps[0], q, D, N, bh) || !make_byte_map(&maps[1], k, D, N, bh) ||
        !make_byte_map(&maps[2], v_t, N, D, bh))
        return FA_ERR_CUDA;
    Params p;
    p.o = o;
    p.lse = lse;
    p.ws_o = nullptr;
    p.ws_st = nullptr;
    p.N = N;
    p.Nk = N;
    p.q_per = N;
    p.causal_off = 0;
    p.packed = 0;
    p.BH = bh;
    p.H = H;
    p.kv_group = 1;
    p.n_qblocks = static_cast<int>(n_qblocks);
    p.n_splits = 1;
    p.n_tiles = static_cast<int>(n_qblocks * BH);
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.q_scale = q_scale;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.n_blocks = n_blocks;
    p.fault_item = -1;
    const cudaError_t e = causal ? launch<128, true, true, false, true>(maps[0], maps[1], maps[2], p, stream)
                                 : launch<128, true, false, false, true>(maps[0], maps[1], maps[2], p, stream);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// ------------------------------------------------------------------ no-allocation split-K
//
// Some callers cannot allocate device memory around this call: a host
// framework that owns every device allocation and hands the library only its
// tensors, or a latency-critical loop in which cudaMalloc / cudaFree (which can
// synchronise the whole device) are not allowed.  For them the split-K pass can
// use a scratch buffer that lives in this library for the life of the process:
// a fixed array in device memory, reserved on every GPU that loads the library.
namespace fa103 {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;   // 64 MiB per device

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Id of the current CUDA context, unique within the process (0 if it cannot be
// read).  A device's context is re-created after cudaDeviceReset, and the
// library's module, with g_noalloc_scratch, is then loaded again, possibly at
// another address: the cached address below is valid only for the context it
// was looked up in.
static unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    });
    if (get_current == nullptr || get_id == nullptr) return 0;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    unsigned long long id = 0;
    return get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

// Device address of g_noalloc_scratch on the current device, looked up with
// that device current the first time it is needed in its context and cached
// per device with the context's id.  In host code the array's name is only a
// stand-in for the symbol, so the kernels must be given this address, never
// the name.
static int noalloc_scratch(void** out) {
    struct Entry {
        unsigned long long ctx_id;
        void* ptr;
    };
    static Entry cache[64];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    const bool cached_dev = dev >= 0 && dev < 64;
    unsigned long long id = current_context_id();
    if (cached_dev && id != 0) {
        std::lock_guard<std::mutex> lock(mu);
        if (cache[dev].ctx_id == id && cache[dev].ptr != nullptr) {
            *out = cache[dev].ptr;
            return FA_OK;
        }
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return FA_ERR_CUDA;
    id = current_context_id();   // the look-up makes the device's context current if it was not yet
    if (cached_dev && id != 0) {
        std::lock_guard<std::mutex> lock(mu);
        cache[dev] = Entry{id, p};
    }
    *out = p;
    return FA_OK;
}

}  // namespace fa103

extern "C" size_t fa_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                      int H, int N, int D, float scale, int causal, int dtype, int num_splits,
                                      cudaStream_t stream) {
    if (num_splits < 1 || num_splits > kMaxSplits) return FA_ERR_INVALID_ARG;
    // Every argument is checked before the scratch address is looked up (the
    // first CUDA call), so bad arguments give the same status as fa_fwd_splitkv.
    const int bad = check_args(q, k, v, o, lse, B, H, H, N, N, D, scale, causal, dtype, num_splits, false);
    if (bad != FA_OK) return bad;
    if (fa_splitkv_workspace_bytes(B, H, N, D, num_splits) > kNoAllocScratchBytes) return FA_ERR_TOO_LARGE;
    void* scratch = nullptr;
    const int st = noalloc_scratch(&scratch);
    if (st != FA_OK) return st;
    return fa_fwd_splitkv(q, k, v, o, lse, B, H, N, D, scale, causal, dtype, num_splits, scratch,
                          kNoAllocScratchBytes, stream);
}

extern "C" int fa_selftest_fwd_fault(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                     int N, int D, float scale, int causal, int dtype, int fault_item,
                                     cudaStream_t stream) {
    if (fault_item < 0) return FA_ERR_INVALID_ARG;
    CUtensorMap maps[3];
    Params p;
    const int st = prepare(q, k, v, o, lse, B, H, H, N, N, D, scale, causal, dtype, 1, false, maps, p);
    if (st != FA_OK) return st;
    p.fault_item = fault_item;
    return dispatch<false>(maps, p, D, dtype, causal, stream);
}

extern "C" int fa_selftest_wait_timeout(cudaStream_t stream) {
    selftest_wait_timeout_kernel<<<1, 32, 0, stream>>>();
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

extern "C" int fa_get_device_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
    unsigned int v = 0, vb = 0;
    if (cudaMemcpyFromSymbol(&v, g_fa_status, sizeof v) != cudaSuccess) return FA_ERR_CUDA;
    if (bwd_take_status(&vb) != 0) return FA_ERR_CUDA;
    if (v != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_fa_status, &zero, sizeof zero) != cudaSuccess) return FA_ERR_CUDA;
    }
    if (vb & kBwdStatusLayout) return FA_ERR_CUDA;
    return (v | vb) != 0 ? FA_ERR_TIMEOUT : FA_OK;
}

extern "C" const char* fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
        case FA_ERR_TOO_LARGE: return "FA_ERR_TOO_LARGE";
        default: return "FA_ERR_UNKNOWN";
    }
}
