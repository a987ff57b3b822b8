// Internal declarations shared by the libgdn translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/gdn.h"

namespace gdn {

constexpr int kChunk = 64;  // prefill chunk grid, tokens

struct DecodeArgs {
    int32_t num_rows, h_k, h_v;
    float scale;
    const uint16_t *q, *k, *v;
    const float *g, *beta;
    float *state;
    int64_t num_slots;
    const int32_t *src_slot, *dst_slot;
    uint16_t *o;
    int32_t *dev_status;
    // Fused input preparation (when a_raw is set): q, k are raw and are
    // normalised in the kernel; g, beta come from a_raw, b_raw, A_log, dt_bias.
    const float *a_raw, *b_raw, *A_log, *dt_bias;
    float eps;
};

// Standalone input preparation.
struct PrepArgs {
    int64_t num_tokens;
    int32_t h_k, h_v;
    const uint16_t *q_raw, *k_raw;
    const float *a, *b, *A_log, *dt_bias;
    float eps;
    uint16_t *q, *k;
    float *g, *beta;
};

// Multi-token decode: tokens_per_row consecutive tokens per row.
struct DecodeMultiArgs {
    int32_t num_rows, tokens_per_row, h_k, h_v;
    float scale;
    const uint16_t *q, *k, *v;  // token t of row r at index r * tokens_per_row + t
    const float *g, *beta;
    float *state;
    int64_t num_slots;
    const int32_t *src_slot;   // [num_rows]
    const int32_t *dst_slots;  // [num_rows * tokens_per_row] or null
    uint16_t *o;
    int32_t *dev_status;
};

struct PrefillArgs {
    int32_t num_seqs, h_k, h_v;
    float scale;
    const int32_t *cu_seqlens;
    const uint16_t *q, *k, *v;
    const float *g, *beta;
    float *state;
    int64_t num_slots;
    const int32_t *src_slot, *dst_slot;
    uint16_t *o;
    float *chunk_states;
    int32_t emit_every_chunks;
    int32_t *dev_status;
    int64_t total_tokens;    // rows of q, k, v, g, beta, o
    int64_t chunk_capacity;  // entries of chunk_states
    // Emission into cache blocks (instead of chunk_states) when emit_table is
    // set: emission k of sequence s goes to slot
    // emit_table[s * emit_table_stride + emit_first[s] + k].
    const int32_t *emit_table;
    const int32_t *emit_first;
    int32_t emit_table_stride;
};

// Launch parameters that depend only on the device (SM count) or on a kernel
// and the device (blocks per SM) are queried once per device and kept for the
// life of the process, so a call costs no attribute or occupancy query.
constexpr int kMaxDevices = 64;
// Current device and its SM count; false if a query failed.
bool current_device(int *dev, int *sms);
// Blocks per SM of `kernel` at `threads` threads and `dyn_smem` bytes of
// dynamic shared memory on device `dev`, cached in `cache` (one slot per device).
template <typename Kernel>
int blocks_per_sm(Kernel kernel, int threads, int dev, int (&cache)[kMaxDevices], size_t dyn_smem = 0) {
    if (dev >= 0 && dev < kMaxDevices && __atomic_load_n(&cache[dev], __ATOMIC_ACQUIRE) > 0)
        return cache[dev];
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, dyn_smem) != cudaSuccess || n < 1) n = 1;
    if (dev >= 0 && dev < kMaxDevices) __atomic_store_n(&cache[dev], n, __ATOMIC_RELEASE);
    return n;
}

// Launchers (decode.cu, prefill.cu).  Arguments are validated by the caller.
cudaError_t launch_decode(const DecodeArgs &a, int d, cudaStream_t stream);
cudaError_t launch_decode_multi(const DecodeMultiArgs &a, int d, cudaStream_t stream);
cudaError_t launch_prep(const PrepArgs &a, int d, cudaStream_t stream);
// cu_host: host mirror of a.cu_seqlens (sizes the launch and orders the chains).
cudaError_t launch_prefill(const PrefillArgs &a, int d, const int32_t *cu_host, cudaStream_t stream);

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&h);
}

// Sum over the 8 lanes of an aligned lane octet; every lane of the octet gets
// the same bits (xor butterfly, each level adds two commuted partial sums).
__device__ __forceinline__ float octet_sum(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    return x;
}

__device__ __forceinline__ void report(int32_t *dev_status, int32_t bit) {
    if (dev_status) atomicOr(dev_status, bit);
}

// Self-checks for debugging builds (-DGDN_DEBUG_CHECKS): a failed check
// records (site, value) of the first failure in dev_status[1..3], sets bit
// 0x100 of dev_status[0], and the guarded access is skipped.  In normal
// builds the guard is the constant true.
#ifdef GDN_DEBUG_CHECKS
__device__ __forceinline__ bool debug_guard(bool ok, int32_t *st, int site, long long val) {
    if (!ok && st) {
        if (atomicCAS(st + 1, 0, site) == 0) {
            st[2] = static_cast<int32_t>(val);
            st[3] = static_cast<int32_t>(val >> 32);
        }
        atomicOr(st, 0x100);
        __threadfence_system();
    }
    return ok;
}
#define GDN_GUARD(st, cond, site, val) ::gdn::debug_guard((cond), (st), (site), static_cast<long long>(val))
#else
#define GDN_GUARD(st, cond, site, val) true
#endif

}  // namespace gdn
