// fa_host.cuh -- host-side helpers shared by the forward and backward
// translation units: tensor-map encoding, SM count, overlap test, and the
// backward pass's device status word (read by fa_get_device_status).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "fa.h"

namespace fa103 {

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn_ptr = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn_ptr = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return fn_ptr;
}

// [BH, N, D] view of a contiguous 16-bit tensor, 128-row x 64-column boxes
// with the 128-byte swizzle.
inline bool make_tile_map(CUtensorMap* map, const void* base, int dtype, int D, int N, int BH) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(N) * D * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t elem_strides[3] = {1, 1, 1};
    CUresult r = enc(map, dtype == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                     const_cast<void*>(base), dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Streaming multiprocessors of a device (cached per device).
inline int sm_count(int dev) {
    static std::atomic<int> cache[64];
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load();
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return -1;
    if (dev >= 0 && dev < 64) cache[dev].store(n);
    return n;
}

inline bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Status bits of the backward kernels on the current device since the last
// call, cleared by the call (0 on success of the read; -1 if CUDA failed).
int bwd_take_status(unsigned int* bits);
// The backward kernel's bit for "shared memory not laid out as required".
constexpr unsigned int kBwdStatusLayout = 64u;

// fa_fwd on H planes that are part of a B = 1 problem of `whole_planes` planes,
// with the forward's form (256-row tiles or the key split) chosen for the whole
// problem, so that per-part results equal the whole call's bit for bit.
int fwd_part(const void* q, const void* k, const void* v, void* o, float* lse, int H, int N, int D, float scale,
             int causal, int dtype, long long whole_planes, cudaStream_t stream);

}  // namespace fa103
