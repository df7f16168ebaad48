// fa_host_io.cu -- the forward pass on host-resident tensors.
//
// Q, K, V live in page-locked host memory and O, LSE are wanted there too.
// The (b, h) planes are cut into chunks; chunk c's inputs are copied to the
// device on one stream, its forward pass runs on the caller's stream as soon as
// they have landed, and its outputs are copied back on a third stream, so the
// copies in both directions overlap the kernel and each other.  Every plane is
// computed by the same kernel as fa_fwd, so the results are bit-identical to
// fa_fwd on the same inputs.

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
    cudaEvent_t start = nullptr, done = nullptr;
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
                  cudaEventCreateWithFlags(&s.done, ev) == cudaSuccess;
        for (int c = 0; ok && c < kMaxChunks; ++c)
            ok = cudaEventCreateWithFlags(&s.in[c], ev) == cudaSuccess &&
                 cudaEventCreateWithFlags(&s.out[c], ev) == cudaSuccess;
        if (!ok) {   // undo, so that a later call starts from nothing
            for (cudaEvent_t* e : {&s.start, &s.done})
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
    for (const void* ptr : {q, k, v, static_cast<const void*>(o), static_cast<const void*>(lse)})
        if (!is_pinned_host(ptr)) return FA_ERR_INVALID_ARG;
    cudaPointerAttributes wa;
    if (cudaPointerGetAttributes(&wa, workspace) != cudaSuccess || wa.type != cudaMemoryTypeDevice) {
        cudaGetLastError();
        return FA_ERR_INVALID_ARG;
    }

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_io_mutex);
    HostIo* io = nullptr;
    const int st0 = io_state(dev, &io);
    if (st0 != FA_OK) return st0;

    // Chunks of whole (b, h) planes: at most kMaxChunks, none much under 8 MiB
    // of inputs, and each with at least kMinChunkTiles work tiles of 256 query
    // rows, so that a chunk's kernel still fills most of the GPU (measured on
    // GB300: fewer, fuller chunks win once a chunk's kernel outlasts its copy).
    const long long planes = static_cast<long long>(B) * H;
    const size_t plane_bytes = L.tensor / static_cast<size_t>(planes);
    long long n_chunks = static_cast<long long>((3 * L.tensor) / kMinChunkBytes);
    const long long by_tiles = planes * ((N + 255) / 256) / kMinChunkTiles;
    if (n_chunks > by_tiles) n_chunks = by_tiles;
    n_chunks = n_chunks < 1 ? 1 : (n_chunks > kMaxChunks ? kMaxChunks : n_chunks);
    if (n_chunks > planes) n_chunks = planes;
    // Chunk starts keep the LSE rows 16-byte aligned: per * N a multiple of 4.
    const long long g = (N % 4 == 0) ? 1 : (N % 2 == 0 ? 2 : 4);
    long long per = (planes + n_chunks - 1) / n_chunks;
    per = (per + g - 1) / g * g;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const uint8_t* hq = static_cast<const uint8_t*>(q);
    const uint8_t* hk = static_cast<const uint8_t*>(k);
    const uint8_t* hv = static_cast<const uint8_t*>(v);
    uint8_t* ho = static_cast<uint8_t*>(o);
    uint8_t* hl = reinterpret_cast<uint8_t*>(lse);
    const size_t lse_plane = static_cast<size_t>(N) * 4;

    bool ok = cudaEventRecord(io->start, stream) == cudaSuccess &&
              cudaStreamWaitEvent(io->h2d, io->start, 0) == cudaSuccess &&
              cudaStreamWaitEvent(io->d2h, io->start, 0) == cudaSuccess;
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
        status = fa_fwd(ws + off, ws + L.k + off, ws + L.v + off, ws + L.o + off,
                        reinterpret_cast<float*>(ws + L.lse + loff), 1, static_cast<int>(np), N, D, scale, causal,
                        dtype, stream);
        ok = status == FA_OK && cudaEventRecord(io->out[c], stream) == cudaSuccess &&
             cudaStreamWaitEvent(io->d2h, io->out[c], 0) == cudaSuccess &&
             cudaMemcpyAsync(ho + off, ws + L.o + off, len, cudaMemcpyDeviceToHost, io->d2h) == cudaSuccess &&
             cudaMemcpyAsync(hl + loff, ws + L.lse + loff, llen, cudaMemcpyDeviceToHost, io->d2h) == cudaSuccess;
        if (!ok && status == FA_OK) status = FA_ERR_CUDA;
    }
    // The caller's stream is ordered after every copy back, also on an error
    // part-way through (what was queued still completes before later work).
    if (cudaEventRecord(io->done, io->d2h) != cudaSuccess || cudaStreamWaitEvent(stream, io->done, 0) != cudaSuccess)
        status = FA_ERR_CUDA;
    return status;
}
