// The small kernels around decode attention:
//   - cache write: slot-mapping scatter of this step's K/V into the block pool
//     (bf16 pools: a copy; FP8 pools: quantised to e4m3 with the pool's scale);
//   - combine: log-sum-exp merge of split-KV partials into bf16 output.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// One thread per 16-byte chunk of a token row.  x indexes
// (token, K|V, chunk) with the chunk fastest, so a warp copies consecutive
// bytes of one row (coalesced 16-byte loads and stores).  A padded slot
// (< 0) is skipped; a slot beyond the pool is skipped and reported.
__global__ void __launch_bounds__(256)
cache_write_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                   const int64_t *__restrict__ slots, int64_t n, uint4 *__restrict__ k_cache,
                   uint4 *__restrict__ v_cache, int64_t n_slots, int row_chunks,
                   int32_t *status) {
    const int64_t total = n * 2 * row_chunks;
    for (int64_t x = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; x < total;
         x += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t c = x % row_chunks;
        const int64_t r = x / row_chunks;  // (token, which)
        const int64_t i = r >> 1;
        const bool is_v = r & 1;
        const int64_t s = slots[i];
        if (s < 0) continue;
        if (s >= n_slots) {
            if (c == 0 && !is_v) set_status(status, PA_STATUS_BAD_SLOT);
            continue;
        }
        const uint4 *src = (is_v ? v_new : k_new) + i * row_chunks + c;
        uint4 *dst = (is_v ? v_cache : k_cache) + s * row_chunks + c;
        *dst = *src;
    }
}

cudaError_t launch_cache_write(const void *k_new, const void *v_new, const int64_t *slots,
                               int64_t n, void *k_cache, void *v_cache, int64_t n_slots,
                               int row_bytes, int32_t *status, cudaStream_t stream) {
    const int row_chunks = row_bytes / 16;
    const int64_t total = n * 2 * row_chunks;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 65535LL * 16) blocks = 65535LL * 16;
    cache_write_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
        static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), slots, n,
        static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), n_slots, row_chunks, status);
    return cudaGetLastError();
}

// FP8 pools: each thread quantises 8 bf16 values of a new K or V row (one
// 16-byte chunk) to e4m3 codes (8 bytes): fp32(x) / scale, rounded to
// nearest even, saturating at the largest finite code (+-448), NaN kept.
__global__ void __launch_bounds__(256)
cache_write_fp8_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                       const int64_t *__restrict__ slots, int64_t n, uint2 *__restrict__ k_cache,
                       uint2 *__restrict__ v_cache, int64_t n_slots, int row_chunks, float k_scale,
                       float v_scale, int32_t *status) {
    const int64_t total = n * 2 * row_chunks;
    for (int64_t x = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; x < total;
         x += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t c = x % row_chunks;
        const int64_t r = x / row_chunks;  // (token, which)
        const int64_t i = r >> 1;
        const bool is_v = r & 1;
        const int64_t s = slots[i];
        if (s < 0) continue;
        if (s >= n_slots) {
            if (c == 0 && !is_v) set_status(status, PA_STATUS_BAD_SLOT);
            continue;
        }
        const uint4 in = (is_v ? v_new : k_new)[i * row_chunks + c];
        (is_v ? v_cache : k_cache)[s * row_chunks + c] = e4m3x8_from_bf16(in, is_v ? v_scale : k_scale);
    }
}

cudaError_t launch_cache_write_fp8(const void *k_new, const void *v_new, const int64_t *slots,
                                   int64_t n, void *k_cache, void *v_cache, int64_t n_slots,
                                   int row_elems, float k_scale, float v_scale, int32_t *status,
                                   cudaStream_t stream) {
    const int row_chunks = row_elems / 8;
    const int64_t total = n * 2 * row_chunks;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 65535LL * 16) blocks = 65535LL * 16;
    cache_write_fp8_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
        static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), slots, n,
        static_cast<uint2 *>(k_cache), static_cast<uint2 *>(v_cache), n_slots, row_chunks, k_scale,
        v_scale, status);
    return cudaGetLastError();
}

// One warp per output row (b, h); each lane owns D/32 dims.  The P partial
// LSEs are read once, coalesced (lane i holds partitions i, i+32, ...); the
// warp reduces their max and sum, so lane i then knows the final weight
// exp(lse_p - lse) of its partitions and hands it to the other lanes by
// shuffle while all lanes stream the partial outputs.  The partial loads of
// consecutive partitions are independent, so the unrolled loop keeps several
// in flight.
template <int D>
__global__ void __launch_bounds__(128)
combine_kernel(__nv_bfloat16 *__restrict__ out, float *__restrict__ lse,
               const float *__restrict__ part_o, const float *__restrict__ part_lse, int rows,
               int P) {
    constexpr int kDPL = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * 4 + warp;
    if (row >= rows) return;
    const float *pl = part_lse + static_cast<int64_t>(row) * P;
    float M = -INFINITY;
    for (int i = lane; i < P; i += 32) M = fmaxf(M, pl[i]);
#pragma unroll
    for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float acc[kDPL];
#pragma unroll
    for (int k = 0; k < kDPL; ++k) acc[k] = 0.f;
    float total = -INFINITY;
    if (M != -INFINITY) {
        float z = 0.f;
        for (int i = lane; i < P; i += 32) z += expf(pl[i] - M);
#pragma unroll
        for (int off = 16; off; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        total = M + logf(z);
        const float *po = part_o + static_cast<int64_t>(row) * P * D + lane * kDPL;
        for (int base = 0; base < P; base += 32) {
            const int i = base + lane;
            const float wl = i < P ? expf(pl[i] - total) : 0.f;  // weight of partition i
            const int n = min(32, P - base);
#pragma unroll 4
            for (int j = 0; j < n; ++j) {
                const float w = __shfl_sync(0xffffffffu, wl, j);
                const float *src = po + static_cast<int64_t>(base + j) * D;
                if constexpr (kDPL == 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(src);
                    acc[0] = fmaf(w, v.x, acc[0]);
                    acc[1] = fmaf(w, v.y, acc[1]);
                    acc[2] = fmaf(w, v.z, acc[2]);
                    acc[3] = fmaf(w, v.w, acc[3]);
                } else {
                    const float2 v = *reinterpret_cast<const float2 *>(src);
                    acc[0] = fmaf(w, v.x, acc[0]);
                    acc[1] = fmaf(w, v.y, acc[1]);
                }
            }
        }
    }
    __nv_bfloat16 *o = out + static_cast<int64_t>(row) * D + lane * kDPL;
#pragma unroll
    for (int k = 0; k < kDPL; k += 2)
        *reinterpret_cast<__nv_bfloat162 *>(o + k) = __floats2bfloat162_rn(acc[k], acc[k + 1]);
    if (lse && lane == 0) lse[row] = total;
}

cudaError_t launch_combine(void *out, float *lse, const float *part_o, const float *part_lse,
                           int rows, int P, int D, cudaStream_t stream) {
    const unsigned blocks = static_cast<unsigned>((rows + 3) / 4);
    if (D == 128)
        combine_kernel<128><<<blocks, 128, 0, stream>>>(static_cast<__nv_bfloat16 *>(out), lse,
                                                         part_o, part_lse, rows, P);
    else if (D == 64)
        combine_kernel<64><<<blocks, 128, 0, stream>>>(static_cast<__nv_bfloat16 *>(out), lse,
                                                        part_o, part_lse, rows, P);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace pa
