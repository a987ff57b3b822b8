// Varlen prefill.  First correct path: one CTA per (sequence, value head)
// keeps the fp32 state S^T in registers and steps through the tokens with the
// same per-row arithmetic as the decode kernel (row_update.cuh).  Emission of
// the carried state follows the 64-token chunk grid anchored at the
// sequence's first token (vLLM page "GatedDeltaNet Automatic Prefix Caching",
// section "Purpose").
#include "row_update.cuh"

namespace gdn {
namespace {

constexpr int kPrefillThreads = 256;
constexpr int kWarps = kPrefillThreads / 32;

// Sum over s' < s of floor(L_s' / (64 E)), by the whole block.
__device__ int64_t emit_offset(const int32_t *cu, int s, int E) {
    __shared__ long long part[kWarps];
    long long acc = 0;
    for (int i = threadIdx.x; i < s; i += blockDim.x)
        acc += (cu[i + 1] - cu[i]) / (kChunk * E);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
    __syncthreads();
    long long tot = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) tot += part[w];
    __syncthreads();
    return tot;
}

template <int D>
__global__ void __launch_bounds__(kPrefillThreads)
prefill_recurrent_kernel(const PrefillArgs a) {
    constexpr int V4 = D / 32;
    constexpr int kRowsPerWarp = D / kWarps;
    constexpr int kGroups = kRowsPerWarp / 4;
    const int seq = blockIdx.x / a.h_v;
    const int h = blockIdx.x % a.h_v;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int sub = lane >> 3;
    const int l8 = lane & 7;
    const int t0 = a.cu_seqlens[seq];
    const int L = a.cu_seqlens[seq + 1] - t0;
    const int E = a.emit_every_chunks;
    const int64_t eoff = (E > 0 && a.chunk_states) ? emit_offset(a.cu_seqlens, seq, E) : 0;

    const int src = a.src_slot ? a.src_slot[seq] : -1;
    const int dst = a.dst_slot ? a.dst_slot[seq] : -1;
    if (src >= a.num_slots || dst >= a.num_slots) {
        report(a.dev_status, GDN_DEV_BAD_SLOT);
        for (int64_t e = threadIdx.x; e < static_cast<int64_t>(L) * D; e += blockDim.x)
            a.o[(static_cast<size_t>(t0 + e / D) * a.h_v + h) * D + e % D] = 0;
        return;
    }

    float4 s[kGroups][V4];
#pragma unroll
    for (int i = 0; i < kGroups; ++i) {
        const int j = warp * kRowsPerWarp + i * 4 + sub;
#pragma unroll
        for (int m = 0; m < V4; ++m) {
            if (src >= 0) {
                const float *sp = a.state + (static_cast<size_t>(src) * a.h_v + h) * D * D;
                s[i][m] = __ldcg(reinterpret_cast<const float4 *>(sp + static_cast<size_t>(j) * D +
                                                                  4 * (l8 + 8 * m)));
            } else {
                s[i][m] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    }

    const int kh = h / (a.h_v / a.h_k);
    for (int t = 0; t < L; ++t) {
        const size_t tok = static_cast<size_t>(t0 + t);
        float kk[V4 * 4], qq[V4 * 4];
        load_bf16_slice<V4>(a.k + (tok * a.h_k + kh) * D, l8, kk);
        load_bf16_slice<V4>(a.q + (tok * a.h_k + kh) * D, l8, qq);
        const size_t gh = tok * a.h_v + h;
        const float alpha = expf(a.g[gh]);
        const float beta = a.beta[gh];
        const float kq = octet_dot<V4>(kk, qq);
        const uint16_t *vrow = a.v + gh * D;
        uint16_t *orow = a.o + gh * D;
#pragma unroll
        for (int i = 0; i < kGroups; ++i) {
            const int j = warp * kRowsPerWarp + i * 4 + sub;
            const float oj = update_row<V4>(s[i], kk, qq, alpha, beta, bf16_bits_to_float(vrow[j]),
                                            kq, a.scale);
            if (l8 == 0) orow[j] = float_to_bf16_bits(oj);
        }
        if (E > 0 && a.chunk_states && ((t + 1) % (kChunk * E)) == 0) {
            const int64_t idx = eoff + (t + 1) / (kChunk * E) - 1;
            float *ep = a.chunk_states + (static_cast<size_t>(idx) * a.h_v + h) * D * D;
#pragma unroll
            for (int i = 0; i < kGroups; ++i) {
                const int j = warp * kRowsPerWarp + i * 4 + sub;
#pragma unroll
                for (int m = 0; m < V4; ++m)
                    __stcg(reinterpret_cast<float4 *>(ep + static_cast<size_t>(j) * D + 4 * (l8 + 8 * m)),
                           s[i][m]);
            }
        }
    }

    if (dst >= 0) {
        float *dp = a.state + (static_cast<size_t>(dst) * a.h_v + h) * D * D;
#pragma unroll
        for (int i = 0; i < kGroups; ++i) {
            const int j = warp * kRowsPerWarp + i * 4 + sub;
#pragma unroll
            for (int m = 0; m < V4; ++m)
                __stcg(reinterpret_cast<float4 *>(dp + static_cast<size_t>(j) * D + 4 * (l8 + 8 * m)),
                       s[i][m]);
        }
    }
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, int d, int64_t total_tokens, int32_t max_seqlen,
                           cudaStream_t stream) {
    (void)total_tokens;
    (void)max_seqlen;
    if (a.num_seqs == 0) return cudaSuccess;
    const int grid = a.num_seqs * a.h_v;
    if (d == 128)
        prefill_recurrent_kernel<128><<<grid, kPrefillThreads, 0, stream>>>(a);
    else
        prefill_recurrent_kernel<64><<<grid, kPrefillThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace gdn
