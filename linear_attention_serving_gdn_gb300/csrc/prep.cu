// Input preparation of the layer ahead of the recurrence: q, k normalised
// per (token, key head) and the decay / write strength formed from raw
// projections (formulas and their fixed evaluation order in row_update.cuh).
// The pages give no formula for this step; the reading is the Gated DeltaNet
// layer's.  Rows are handled by lane octets in exactly the decode kernel's
// layout, so this kernel followed by gdn_decode_packed equals the fused
// gdn_decode_packed_raw bit for bit.  Memory-bound: one read and one write of
// q, k, and a, b -> g, beta.
#include "row_update.cuh"

namespace gdn {
namespace {

constexpr int kPrepThreads = 256;

template <int D>
__global__ void __launch_bounds__(kPrepThreads, 5) prep_kernel(const PrepArgs a) {
    constexpr int V4 = D / 32;
    const int lane = threadIdx.x & 31;
    const int sub = lane >> 3, l8 = lane & 7;
    const int64_t rows_per_tensor = a.num_tokens * a.h_k;
    const int64_t rows = 2 * rows_per_tensor;  // q rows, then k rows
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    // Warp-uniform loop over 8 rows at a time, two groups of 4 (one row per
    // lane octet), both groups' loads issued before either reduction: every
    // lane takes part in the octet reductions; octets past the end only skip
    // I/O.
    for (int64_t base = warp * 8; base < rows; base += nwarps * 8) {
        float x[2][V4 * 4];
        bool live[2], is_k[2];
        int64_t rr[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t row = base + 4 * u + sub;
            live[u] = row < rows;
            is_k[u] = row >= rows_per_tensor;
            rr[u] = is_k[u] ? row - rows_per_tensor : row;
            if (live[u]) {
                load_bf16_slice<V4>((is_k[u] ? a.k_raw : a.q_raw) + rr[u] * D, l8, x[u]);
            } else {
#pragma unroll
                for (int e = 0; e < V4 * 4; ++e) x[u][e] = 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            normalize_bf16<V4>(x[u], a.eps);
            if (live[u]) store_bf16_slice<V4>((is_k[u] ? a.k : a.q) + rr[u] * D, l8, x[u]);
        }
    }
    // Gates: a, b -> g, beta over the flat [token][value head] arrays.  With
    // 16-byte aligned arrays each thread takes runs of four elements (float4
    // loads and stores), kGateRuns runs at a time with all their loads issued
    // first while whole sets remain, then single runs; the last n_gate % 4
    // elements, and unaligned arrays, go one element at a time.  The head of
    // element e is e % h_v, stepped by the stride's residue.
    const int64_t n_gate = a.num_tokens * a.h_v;
    const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const bool vec = ((reinterpret_cast<uintptr_t>(a.a) | reinterpret_cast<uintptr_t>(a.b) |
                       reinterpret_cast<uintptr_t>(a.g) | reinterpret_cast<uintptr_t>(a.beta)) & 15u) == 0;
    int64_t done = 0;  // elements [0, done) are handled by the vector loops
    if (vec) {
        constexpr int kGateRuns = 2;
        const int64_t n4 = n_gate / 4;  // runs of four
        const int dh = static_cast<int>((4 * nthreads) % a.h_v);
        auto adv = [&](int hh, int d) {
            hh += d;
            return hh >= a.h_v ? hh - a.h_v : hh;
        };
        auto run = [&](int64_t j, float4 av, float4 bv, int h) {
            float4 gv, btv;
            gate_inputs(av.x, bv.x, a.A_log[h], a.dt_bias[h], gv.x, btv.x);
            h = adv(h, 1);
            gate_inputs(av.y, bv.y, a.A_log[h], a.dt_bias[h], gv.y, btv.y);
            h = adv(h, 1);
            gate_inputs(av.z, bv.z, a.A_log[h], a.dt_bias[h], gv.z, btv.z);
            h = adv(h, 1);
            gate_inputs(av.w, bv.w, a.A_log[h], a.dt_bias[h], gv.w, btv.w);
            reinterpret_cast<float4 *>(a.g)[j] = gv;
            reinterpret_cast<float4 *>(a.beta)[j] = btv;
        };
        int64_t j = tid;
        int h = static_cast<int>((4 * j) % a.h_v);
        for (; j + (kGateRuns - 1) * nthreads < n4; j += kGateRuns * nthreads) {
            float4 av[kGateRuns], bv[kGateRuns];
#pragma unroll
            for (int u = 0; u < kGateRuns; ++u) {
                av[u] = reinterpret_cast<const float4 *>(a.a)[j + u * nthreads];
                bv[u] = reinterpret_cast<const float4 *>(a.b)[j + u * nthreads];
            }
#pragma unroll
            for (int u = 0; u < kGateRuns; ++u) {
                run(j + u * nthreads, av[u], bv[u], h);
                h = adv(h, dh);
            }
        }
        for (; j < n4; j += nthreads, h = adv(h, dh))
            run(j, reinterpret_cast<const float4 *>(a.a)[j], reinterpret_cast<const float4 *>(a.b)[j], h);
        done = 4 * n4;
    }
    for (int64_t e = done + tid; e < n_gate; e += nthreads) {
        const int h = static_cast<int>(e % a.h_v);
        float g, beta;
        gate_inputs(a.a[e], a.b[e], a.A_log[h], a.dt_bias[h], g, beta);
        a.g[e] = g;
        a.beta[e] = beta;
    }
}

template <int D>
cudaError_t launch_prep_d(const PrepArgs &a, cudaStream_t stream) {
    static int occ[kMaxDevices] = {};
    int dev = 0, sms = 0;
    if (!current_device(&dev, &sms)) return cudaErrorInvalidDevice;
    const int64_t rows = 2 * a.num_tokens * a.h_k;
    const int64_t need_rows = (rows + (kPrepThreads / 4) - 1) / (kPrepThreads / 4);  // 8 rows per warp
    const int64_t need_gate = (a.num_tokens * a.h_v + kPrepThreads - 1) / kPrepThreads;
    int64_t grid = need_rows > need_gate ? need_rows : need_gate;
    // One wave of resident blocks: every block walks the rows with the same
    // grid stride, so blocks beyond the resident count would run as a short,
    // half-empty second wave.
    const int64_t cap = static_cast<int64_t>(sms) * blocks_per_sm(prep_kernel<D>, kPrepThreads, dev, occ);
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    prep_kernel<D><<<static_cast<int>(grid), kPrepThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prep(const PrepArgs &a, int d, cudaStream_t stream) {
    if (a.num_tokens == 0) return cudaSuccess;
    return d == 128 ? launch_prep_d<128>(a, stream) : launch_prep_d<64>(a, stream);
}

}  // namespace gdn
