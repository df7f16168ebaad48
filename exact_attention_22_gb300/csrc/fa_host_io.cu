// fa_host_io.cu -- the forward (16-bit and FP8) and backward passes on
// host-resident tensors.
//
// The inputs live in page-locked host memory and the outputs are wanted there
// too.  The (b, h) planes are cut into chunks; chunk c's inputs are copied to
// the device on one stream, its pass (fa_fwd, fa_fwd_fp8 or fa_bwd on the
// chunk's planes) runs on the caller's stream as soon as they have landed, and
// its outputs are copied back on a third stream, so the copies in both
// directions overlap the kernels and each other.  Every plane is computed by the
// same kernels as the device entry points.

#include <cmath>
#include <cstddef>
#include <cstdint>
#include <initializer_list>
#include <mutex>

#include "fa_host.cuh"

namespace fa103 {
namespace {

constexpr int kMaxChunks = 8;
constexpr size_t kMinChunkBytes = size_t(8) << 20;   // below this a chunk's copy is launch-bound
constexpr long long kMinChunkTiles = 128;

// Per-device copy streams and events, created on first use and kept for the
// life of the process (like a library handle).
struct HostIo {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, done = nullptr, in_done = nullptr;
    cudaEvent_t in[kMaxChunks] = {}, out[kMaxChunks] = {};
};

std::mutex g_io_mutex;   // one enqueue at a time: the streams and events are shared
HostIo g_io[64];

int io_state(int dev, HostIo** out) {
    if (dev < 0 || dev >= 64) return FA_ERR_UNSUPPORTED;
    HostIo& s = g_io[dev];
    if (!s.ready) {
        const unsigned ev = cudaEventDisableTiming;
        bool ok = cudaStreamCreateWithFlags(&s.h2d, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&s.d2h, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&s.start, ev) == cudaSuccess &&
                  cudaEventCreateWithFlags(&s.done, ev) == cudaSuccess &&
                  cudaEventCreateWithFlags(&s.in_done, ev) == cudaSuccess;
        for (int c = 0; ok && c < kMaxChunks; ++c)
            ok = cudaEventCreateWithFlags(&s.in[c], ev) == cudaSuccess &&
                 cudaEventCreateWithFlags(&s.out[c], ev) == cudaSuccess;
        if (!ok) {   // undo, so that a later call starts from nothing
            for (cudaEvent_t* e : {&s.start, &s.done, &s.in_done})
                if (*e) cudaEventDestroy(*e), *e = nullptr;
            for (int c = 0; c < kMaxChunks; ++c) {
                if (s.in[c]) cudaEventDestroy(s.in[c]), s.in[c] = nullptr;
                if (s.out[c]) cudaEventDestroy(s.out[c]), s.out[c] = nullptr;
            }
            for (cudaStream_t* t : {&s.h2d, &s.d2h})
                if (*t) cudaStreamDestroy(*t), *t = nullptr;
            return FA_ERR_CUDA;
        }
        s.ready = true;
    }
    *out = &s;
    return FA_OK;
}

bool is_pinned_host(const void* ptr) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Planes per chunk: at most kMaxChunks chunks, none much under 8 MiB of inputs,
// and each with at least kMinChunkTiles work tiles (of `tile_rows` rows of a
// plane), so that a chunk's kernel still fills most of the GPU (measured on
// GB300: fewer, fuller chunks win once a chunk's kernel outlasts its copy).
// Chunk starts keep the LSE rows 16-byte aligned: planes per chunk times N is
// a multiple of 4.
long long chunk_planes(long long planes, int N, size_t in_bytes, int tile_rows) {
    long long n_chunks = static_cast<long long>(in_bytes / kMinChunkBytes);
    const long long by_tiles = planes * ((N + tile_rows - 1) / tile_rows) / kMinChunkTiles;
    if (n_chunks > by_tiles) n_chunks = by_tiles;
    n_chunks = n_chunks < 1 ? 1 : (n_chunks > kMaxChunks ? kMaxChunks : n_chunks);
    if (n_chunks > planes) n_chunks = planes;
    const long long g = (N % 4 == 0) ? 1 : (N % 2 == 0 ? 2 : 4);
    const long long per = (planes + n_chunks - 1) / n_chunks;
    return (per + g - 1) / g * g;
}

// Checks shared by the host entry points: every host buffer page-locked, the
// workspace device memory.
bool host_buffers_ok(std::initializer_list<const void*> host, const void* workspace) {
    for (const void* ptr : host)
        if (!is_pinned_host(ptr)) return false;
    cudaPointerAttributes wa;
    if (cudaPointerGetAttributes(&wa, workspace) != cudaSuccess || wa.type != cudaMemoryTypeDevice) {
        cudaGetLastError();
        return false;
    }
    return true;
}

// Copy streams ordered after the work already queued on `stream`.
bool pipeline_begin(HostIo* io, cudaStream_t stream) {
    return cudaEventRecord(io->start, stream) == cudaSuccess &&
           cudaStreamWaitEvent(io->h2d, io->start, 0) == cudaSuccess &&
           cudaStreamWaitEvent(io->d2h, io->start, 0) == cudaSuccess;
}

// `stream` ordered after every copy in both directions, also after an error
// part-way through: a chunk's inputs may be queued when its kernel fails to
// launch, and those copies still use the caller's buffers.
bool pipeline_end(HostIo* io, cudaStream_t stream) {
    return cudaEventRecord(io->in_done, io->h2d) == cudaSuccess &&
           cudaStreamWaitEvent(stream, io->in_done, 0) == cudaSuccess &&
           cudaEventRecord(io->done, io->d2h) == cudaSuccess && cudaStreamWaitEvent(stream, io->done, 0) == cudaSuccess;
}

// Device workspace: Q, K, V, O ([B,H,N,D] 16-bit each), then LSE ([B,H,N] fp32).
struct Layout {
    size_t tensor, lse_bytes, k, v, o, lse, total;
};

bool layout(int B, int H, int N, int D, Layout* L) {
    if (B < 1 || H < 1 || N < 1 || (D != 64 && D != 128)) return false;
    const uint64_t elems = static_cast<uint64_t>(B) * static_cast<uint64_t>(H) * static_cast<uint64_t>(N) * D;
    if (elems >= (uint64_t(1) << 40)) return false;
    L->tensor = static_cast<size_t>(elems) * 2;
    L->lse_bytes = static_cast<size_t>(elems / D) * 4;
    L->k = align256(L->tensor);
    L->v = 2 * L->k;
    L->o = 3 * L->k;
    L->lse = 4 * L->k;
    L->total = L->lse + align256(L->lse_bytes);
    return true;
}

}  // namespace
}  // namespace fa103

using namespace fa103;

extern "C" size_t fa_fwd_host_workspace_bytes(int B, int H, int N, int D) {
    Layout L;
    return layout(B, H, N, D, &L) ? L.total : 0;
}

extern "C" int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                           int D, float scale, int causal, int dtype, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
    // The argument rules of fa_fwd, checked here so that nothing is queued on
    // an error.
    if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    Layout L;
    if (!layout(B, H, N, D, &L)) return FA_ERR_INVALID_ARG;
    const void* ptrs[6] = {q, k, v, o, lse, workspace};
    for (const void* ptr : ptrs)
        if (ptr == nullptr || (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0) return FA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_MISALIGNED;
    if (workspace_bytes < L.total) return FA_ERR_INVALID_ARG;
    const void* ins[3] = {q, k, v};
    for (const void* in : ins)
        if (overlaps(o, L.tensor, in, L.tensor) || overlaps(lse, L.lse_bytes, in, L.tensor)) return FA_ERR_INVALID_ARG;
    if (overlaps(o, L.tensor, lse, L.lse_bytes)) return FA_ERR_INVALID_ARG;
    if (!host_buffers_ok({q, k, v, o, lse}, workspace)) return FA_ERR_INVALID_ARG;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_io_mutex);
    HostIo* io = nullptr;
    const int st0 = io_state(dev, &io);
    if (st0 != FA_OK) return st0;

    // Chunks of whole (b, h) planes; the forward's work tiles are 256 query rows.
    const long long planes = static_cast<long long>(B) * H;
    const size_t plane_bytes = L.tensor / static_cast<size_t>(planes);
    const long long per = chunk_planes(planes, N, 3 * L.tensor, 256);

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const uint8_t* hq = static_cast<const uint8_t*>(q);
    const uint8_t* hk = static_cast<const uint8_t*>(k);
    const uint8_t* hv = static_cast<const uint8_t*>(v);
    uint8_t* ho = static_cast<uint8_t*>(o);
    uint8_t* hl = reinterpret_cast<uint8_t*>(lse);
    const size_t lse_plane = static_cast<size_t>(N) * 4;

    bool ok = pipeline_begin(io, stream);
    int status = ok ? FA_OK : FA_ERR_CUDA;
    for (int c = 0; ok && c * per < planes; ++c) {
        const long long p0 = c * per, np = (planes - p0 < per) ? planes - p0 : per;
        const size_t off = static_cast<size_t>(p0) * plane_bytes, len = static_cast<size_t>(np) * plane_bytes;
        const size_t loff = static_cast<size_t>(p0) * lse_plane, llen = static_cast<size_t>(np) * lse_plane;
        ok = cudaMemcpyAsync(ws + off, hq + off, len, cudaMemcpyHostToDevice, io->h2d) == cudaSuccess &&
             cudaMemcpyAsync(ws + L.k + off, hk + off, len, cudaMemcpyHostToDevice, io->h2d) == cudaSuccess &&
             cudaMemcpyAsync(ws + L.v + off, hv + off, len, cudaMemcpyHostToDevice, io->h2d) == cudaSuccess &&
             cudaEventRecord(io->in[c], io->h2d) == cudaSuccess &&
             cudaStreamWaitEvent(stream, io->in[c], 0) == cudaSuccess;
        if (!ok) {
            status = FA_ERR_CUDA;
            break;
        }
        status = fwd_part(ws + off, ws + L.k + off, ws + L.v + off, ws + L.o + off,
                          reinterpret_cast<float*>(ws + L.lse + loff), static_cast<int>(np), N, D, scale, causal,
                          dtype, planes, stream);
        ok = status == FA_OK && cudaEventRecord(io->out[c], stream) == cudaSuccess &&
             cudaStreamWaitEvent(io->d2h, io->out[c], 0) == cudaSuccess &&
             cudaMemcpyAsync(ho + off, ws + L.o + off, len, cudaMemcpyDeviceToHost, io->d2h) == cudaSuccess &&
             cudaMemcpyAsync(hl + loff, ws + L.lse + loff, llen, cudaMemcpyDeviceToHost, io->d2h) == cudaSuccess;
        if (!ok && status == FA_OK) status = FA_ERR_CUDA;
    }
    if (!pipeline_end(io, stream)) status = FA_ERR_CUDA;
    return status;
}

// ------------------------------------------------------------------ backward

namespace fa103 {
namespace {

// Device workspace of fa_bwd_host: Q, K, V, O, dO, dQ, dK, dV ([B,H,N,D]
// 16-bit each), the LSE ([B,H,N] fp32), then fa_bwd's own workspace for one
// chunk (reused by the chunks in turn: they run one after another on the
// caller's stream).
struct BwdLayout {
    size_t tensor, lse_bytes, stride, lse, bws, bws_bytes, total;
    long long per;
};

bool bwd_layout(int B, int H, int N, int D, BwdLayout* L) {
    if (B < 1 || H < 1 || N < 1 || (D != 64 && D != 128)) return false;
    const uint64_t planes = static_cast<uint64_t>(B) * static_cast<uint64_t>(H);
    const uint64_t elems = planes * static_cast<uint64_t>(N) * D;
    if (planes > 0x7fffffffull || elems >= (uint64_t(1) << 40)) return false;
    L->tensor = static_cast<size_t>(elems) * 2;
    L->lse_bytes = static_cast<size_t>(elems / D) * 4;
    L->stride = align256(L->tensor);
    L->lse = 8 * L->stride;
    L->per = chunk_planes(static_cast<long long>(planes), N, 5 * L->tensor, 128);
    L->bws = L->lse + align256(L->lse_bytes);
    L->bws_bytes = fa_bwd_workspace_bytes(1, static_cast<int>(L->per), N, D);
    if (L->bws_bytes == 0) return false;
    L->total = L->bws + L->bws_bytes;
    return true;
}

}  // namespace
}  // namespace fa103

extern "C" size_t fa_bwd_host_workspace_bytes(int B, int H, int N, int D) {
    BwdLayout L;
    return bwd_layout(B, H, N, D, &L) ? L.total : 0;
}

extern "C" int fa_bwd_host(const void* q, const void* k, const void* v, const void* o, const void* dout,
                           const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int D, float scale,
                           int causal, int dtype, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    // The argument rules of fa_bwd, checked here so that nothing is queued on
    // an error.
    if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    BwdLayout L;
    if (!bwd_layout(B, H, N, D, &L)) return FA_ERR_INVALID_ARG;
    const void* ptrs[10] = {q, k, v, o, dout, lse, dq, dk, dv, workspace};
    for (const void* ptr : ptrs)
        if (ptr == nullptr || (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0) return FA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_MISALIGNED;
    if (workspace_bytes < L.total) return FA_ERR_INVALID_ARG;
    const void* ins[6] = {q, k, v, o, dout, lse};
    const size_t in_bytes[6] = {L.tensor, L.tensor, L.tensor, L.tensor, L.tensor, L.lse_bytes};
    const void* outs[3] = {dq, dk, dv};
    for (int a = 0; a < 3; ++a) {
        for (int b = 0; b < 6; ++b)
            if (overlaps(outs[a], L.tensor, ins[b], in_bytes[b])) return FA_ERR_INVALID_ARG;
        for (int b = a + 1; b < 3; ++b)
            if (overlaps(outs[a], L.tensor, outs[b], L.tensor)) return FA_ERR_INVALID_ARG;
    }
    if (!host_buffers_ok({q, k, v, o, dout, lse, dq, dk, dv}, workspace)) return FA_ERR_INVALID_ARG;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_io_mutex);
    HostIo* io = nullptr;
    const int st0 = io_state(dev, &io);
    if (st0 != FA_OK) return st0;

    // Chunks of whole (b, h) planes; the backward's work tiles are 128 keys.
    const long long planes = static_cast<long long>(B) * H;
    const size_t plane_bytes = L.tensor / static_cast<size_t>(planes);
    const size_t lse_plane = static_cast<size_t>(N) * 4;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const uint8_t* hin[5] = {static_cast<const uint8_t*>(q), static_cast<const uint8_t*>(k),
                             static_cast<const uint8_t*>(v), static_cast<const uint8_t*>(o),
                             static_cast<const uint8_t*>(dout)};
    uint8_t* hout[3] = {static_cast<uint8_t*>(dq), static_cast<uint8_t*>(dk), static_cast<uint8_t*>(dv)};
    const uint8_t* hl = reinterpret_cast<const uint8_t*>(lse);

    bool ok = pipeline_begin(io, stream);
    int status = ok ? FA_OK : FA_ERR_CUDA;
    for (int c = 0; ok && c * L.per < planes; ++c) {
        const long long p0 = c * L.per, np = (planes - p0 < L.per) ? planes - p0 : L.per;
        const size_t off = static_cast<size_t>(p0) * plane_bytes, len = static_cast<size_t>(np) * plane_bytes;
        const size_t loff = static_cast<size_t>(p0) * lse_plane, llen = static_cast<size_t>(np) * lse_plane;
        for (int t = 0; ok && t < 5; ++t)
            ok = cudaMemcpyAsync(ws + t * L.stride + off, hin[t] + off, len, cudaMemcpyHostToDevice, io->h2d) ==
                 cudaSuccess;
        ok = ok &&
             cudaMemcpyAsync(ws + L.lse + loff, hl + loff, llen, cudaMemcpyHostToDevice, io->h2d) == cudaSuccess &&
             cudaEventRecord(io->in[c], io->h2d) == cudaSuccess &&
             cudaStreamWaitEvent(stream, io->in[c], 0) == cudaSuccess;
        if (!ok) {
            status = FA_ERR_CUDA;
            break;
        }
        status = fa_bwd(ws + off, ws + L.stride + off, ws + 2 * L.stride + off, ws + 3 * L.stride + off,
                        ws + 4 * L.stride + off, reinterpret_cast<const float*>(ws + L.lse + loff),
                        ws + 5 * L.stride + off, ws + 6 * L.stride + off, ws + 7 * L.stride + off, 1,
                        static_cast<int>(np), N, D, scale, causal, dtype, ws + L.bws, L.bws_bytes, stream);
        ok = status == FA_OK && cudaEventRecord(io->out[c], stream) == cudaSuccess &&
             cudaStreamWaitEvent(io->d2h, io->out[c], 0) == cudaSuccess;
        for (int t = 0; ok && t < 3; ++t)
            ok = cudaMemcpyAsync(hout[t] + off, ws + (5 + t) * L.stride + off, len, cudaMemcpyDeviceToHost,
                                 io->d2h) == cudaSuccess;
        if (!ok && status == FA_OK) status = FA_ERR_CUDA;
    }
    if (!pipeline_end(io, stream)) status = FA_ERR_CUDA;
    return status;
}

// ------------------------------------------------------------------ FP8 forward

namespace fa103 {
namespace {

// Device workspace of fa_fwd_fp8_host: Q, K (E4M3 [B,H,N,D]), V^T (E4M3
// [B,H,D,N]), the three block-scale arrays ([B,H,ceil(N/128)] fp32), O (bf16
// [B,H,N,D]) and the LSE ([B,H,N] fp32), each rounded up to 256 bytes.
struct Fp8Layout {
    size_t elems, sc_bytes, o_bytes, lse_bytes, k, vt, qs, ks, vs, o, lse, total;
    int n_blocks;
};

bool fp8_layout(int B, int H, int N, int D, Fp8Layout* L) {
    if (B < 1 || H < 1 || N < 1 || D != 128 || N % 16 != 0) return false;
    const uint64_t planes = static_cast<uint64_t>(B) * static_cast<uint64_t>(H);
    const uint64_t elems = planes * static_cast<uint64_t>(N) * D;
    if (planes > 0x7fffffffull || elems >= (uint64_t(1) << 40)) return false;
    L->n_blocks = (N + 127) / 128;
    L->elems = static_cast<size_t>(elems);
    L->sc_bytes = static_cast<size_t>(planes) * L->n_blocks * 4;
    L->o_bytes = L->elems * 2;
    L->lse_bytes = static_cast<size_t>(planes) * N * 4;
    L->k = align256(L->elems);
    L->vt = L->k + align256(L->elems);
    L->qs = L->vt + align256(L->elems);
    L->ks = L->qs + align256(L->sc_bytes);
    L->vs = L->ks + align256(L->sc_bytes);
    L->o = L->vs + align256(L->sc_bytes);
    L->lse = L->o + align256(L->o_bytes);
    L->total = L->lse + align256(L->lse_bytes);
    return true;
}

}  // namespace
}  // namespace fa103

extern "C" size_t fa_fwd_fp8_host_workspace_bytes(int B, int H, int N, int D) {
    Fp8Layout L;
    return fp8_layout(B, H, N, D, &L) ? L.total : 0;
}

extern "C" int fa_fwd_fp8_host(const void* q, const void* k, const void* v_t, const float* q_scale,
                               const float* k_scale, const float* v_scale, void* o, float* lse, int B, int H, int N,
                               int D, float scale, int causal, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
    // The argument rules of fa_fwd_fp8, checked here so that nothing is queued
    // on an error.
    if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    if (D != 128) return FA_ERR_UNSUPPORTED;
    if (N % 16 != 0) return FA_ERR_INVALID_ARG;
    Fp8Layout L;
    if (!fp8_layout(B, H, N, D, &L)) return FA_ERR_INVALID_ARG;
    const void* ptrs[9] = {q, k, v_t, q_scale, k_scale, v_scale, o, lse, workspace};
    for (const void* ptr : ptrs)
        if (ptr == nullptr || (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0) return FA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_MISALIGNED;
    if (workspace_bytes < L.total) return FA_ERR_INVALID_ARG;
    const void* ins[6] = {q, k, v_t, q_scale, k_scale, v_scale};
    const size_t ib[6] = {L.elems, L.elems, L.elems, L.sc_bytes, L.sc_bytes, L.sc_bytes};
    for (int i = 0; i < 6; ++i)
        if (overlaps(o, L.o_bytes, ins[i], ib[i]) || overlaps(lse, L.lse_bytes, ins[i], ib[i]))
            return FA_ERR_INVALID_ARG;
    if (overlaps(o, L.o_bytes, lse, L.lse_bytes)) return FA_ERR_INVALID_ARG;
    if (!host_buffers_ok({q, k, v_t, q_scale, k_scale, v_scale, o, lse}, workspace)) return FA_ERR_INVALID_ARG;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_io_mutex);
    HostIo* io = nullptr;
    const int st0 = io_state(dev, &io);
    if (st0 != FA_OK) return st0;

    // Chunks of whole planes; chunk starts also keep the block scales 16-byte
    // aligned (planes per chunk times the blocks per plane a multiple of 4).
    const long long planes = static_cast<long long>(B) * H;
    long long per = chunk_planes(planes, N, 3 * L.elems, 256);
    const long long g = (L.n_blocks % 4 == 0) ? 1 : (L.n_blocks % 2 == 0 ? 2 : 4);
    per = (per + g - 1) / g * g;
    const size_t plane_in = L.elems / static_cast<size_t>(planes), plane_sc = static_cast<size_t>(L.n_blocks) * 4;
    const size_t plane_o = plane_in * 2, plane_l = static_cast<size_t>(N) * 4;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const uint8_t* hin[3] = {static_cast<const uint8_t*>(q), static_cast<const uint8_t*>(k),
                             static_cast<const uint8_t*>(v_t)};
    const size_t din[3] = {0, L.k, L.vt};
    const uint8_t* hsc[3] = {reinterpret_cast<const uint8_t*>(q_scale), reinterpret_cast<const uint8_t*>(k_scale),
                             reinterpret_cast<const uint8_t*>(v_scale)};
    const size_t dsc[3] = {L.qs, L.ks, L.vs};

    bool ok = pipeline_begin(io, stream);
    int status = ok ? FA_OK : FA_ERR_CUDA;
    for (int c = 0; ok && c * per < planes; ++c) {
        const long long p0 = c * per, np = (planes - p0 < per) ? planes - p0 : per;
        const size_t p0s = static_cast<size_t>(p0), nps = static_cast<size_t>(np);
        for (int t = 0; ok && t < 3; ++t)
            ok = cudaMemcpyAsync(ws + din[t] + p0s * plane_in, hin[t] + p0s * plane_in, nps * plane_in,
                                 cudaMemcpyHostToDevice, io->h2d) == cudaSuccess &&
                 cudaMemcpyAsync(ws + dsc[t] + p0s * plane_sc, hsc[t] + p0s * plane_sc, nps * plane_sc,
                                 cudaMemcpyHostToDevice, io->h2d) == cudaSuccess;
        ok = ok && cudaEventRecord(io->in[c], io->h2d) == cudaSuccess &&
             cudaStreamWaitEvent(stream, io->in[c], 0) == cudaSuccess;
        if (!ok) {
            status = FA_ERR_CUDA;
            break;
        }
        status = fa_fwd_fp8(ws + p0s * plane_in, ws + L.k + p0s * plane_in, ws + L.vt + p0s * plane_in,
                            reinterpret_cast<const float*>(ws + L.qs + p0s * plane_sc),
                            reinterpret_cast<const float*>(ws + L.ks + p0s * plane_sc),
                            reinterpret_cast<const float*>(ws + L.vs + p0s * plane_sc), ws + L.o + p0s * plane_o,
                            reinterpret_cast<float*>(ws + L.lse + p0s * plane_l), 1, static_cast<int>(np), N, D,
                            scale, causal, stream);
        ok = status == FA_OK && cudaEventRecord(io->out[c], stream) == cudaSuccess &&
             cudaStreamWaitEvent(io->d2h, io->out[c], 0) == cudaSuccess &&
             cudaMemcpyAsync(static_cast<uint8_t*>(o) + p0s * plane_o, ws + L.o + p0s * plane_o, nps * plane_o,
                             cudaMemcpyDeviceToHost, io->d2h) == cudaSuccess &&
             cudaMemcpyAsync(reinterpret_cast<uint8_t*>(lse) + p0s * plane_l, ws + L.lse + p0s * plane_l,
                             nps * plane_l, cudaMemcpyDeviceToHost, io->d2h) == cudaSuccess;
        if (!ok && status == FA_OK) status = FA_ERR_CUDA;
    }
    if (!pipeline_end(io, stream)) status = FA_ERR_CUDA;
    return status;
}
