// Host-side cost of one libgdn call, measured from C (no Python in the path).
//
// Each entry point is called back to back on one stream with a tiny problem
// (one decode row; one 64-token prefill; the two together as a mixed step),
// so the GPU keeps up and the host time per call is the library's own cost:
// argument validation, launch-parameter lookup and the kernel launch.
// Prints one JSON object: microseconds of host time per call.
#include <cuda_runtime.h>

#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "gdn.h"

namespace {

template <typename F>
double us_per_call(F &&call, int n, cudaStream_t st) {
    for (int i = 0; i < 50; ++i) call();
    cudaStreamSynchronize(st);
    const auto t0 = std::chrono::steady_clock::now();
    for (int i = 0; i < n; ++i) call();
    const auto t1 = std::chrono::steady_clock::now();
    cudaStreamSynchronize(st);
    return std::chrono::duration<double, std::micro>(t1 - t0).count() / n;
}

}  // namespace

int main(int argc, char **argv) {
    const int n = argc > 1 ? atoi(argv[1]) : 2000;
    const int H = 16, D = 128, T = 64;
    gdn_dims_t dims{H, H, D, D, 1.0f};
    const size_t act = static_cast<size_t>(T + 1) * H * D;  // one decode row + 64 prefill tokens
    uint16_t *q, *k, *v, *o;
    float *g, *beta, *state;
    int32_t *slots, *cu, *status;
    if (cudaMalloc(&q, act * 2) || cudaMalloc(&k, act * 2) || cudaMalloc(&v, act * 2) || cudaMalloc(&o, act * 2) ||
        cudaMalloc(&g, (T + 1) * H * 4) || cudaMalloc(&beta, (T + 1) * H * 4) ||
        cudaMalloc(&state, 4ull * H * D * D * 4) || cudaMalloc(&slots, 16) || cudaMalloc(&cu, 8) ||
        cudaMalloc(&status, 4)) {
        printf("{\"error\": \"cudaMalloc failed\"}\n");
        return 1;
    }
    cudaMemset(q, 0, act * 2);
    cudaMemset(k, 0, act * 2);
    cudaMemset(v, 0, act * 2);
    cudaMemset(g, 0, (T + 1) * H * 4);
    cudaMemset(beta, 0, (T + 1) * H * 4);
    cudaMemset(state, 0, 4ull * H * D * D * 4);
    const int32_t hslots[4] = {0, 1, 2, 3}, hcu[2] = {0, T};
    cudaMemcpy(slots, hslots, 16, cudaMemcpyHostToDevice);
    cudaMemcpy(cu, hcu, 8, cudaMemcpyHostToDevice);
    cudaStream_t st;
    cudaStreamCreate(&st);
    const size_t row = static_cast<size_t>(H) * D;
    int bad = 0;
    auto decode = [&] {
        bad |= gdn_decode_packed(&dims, 1, q, k, v, g, beta, state, 4, slots, nullptr, o, status, st);
    };
    auto prefill = [&] {
        bad |= gdn_prefill_varlen(&dims, 1, cu, hcu, q + row, k + row, v + row, g + H, beta + H, state, 4, nullptr,
                                  slots + 1, o + row, nullptr, 0, 0, nullptr, 0, status, st);
    };
    auto mixed = [&] {
        bad |= gdn_mixed_step(&dims, 1, 1, cu, hcu, q, k, v, g, beta, state, 4, slots, nullptr, nullptr, slots + 2,
                              o, nullptr, 0, 0, nullptr, 0, status, st);
    };
    const double d_us = us_per_call(decode, n, st);
    const double p_us = us_per_call(prefill, n / 4, st);
    const double m_us = us_per_call(mixed, n / 4, st);
    const cudaError_t e = cudaStreamSynchronize(st);
    printf("{\"decode_packed_us\": %.3f, \"prefill_varlen_us\": %.3f, \"mixed_step_us\": %.3f, \"calls\": %d, "
           "\"ok\": %s}\n",
           d_us, p_us, m_us, n, (bad == 0 && e == cudaSuccess) ? "true" : "false");
    return (bad == 0 && e == cudaSuccess) ? 0 : 1;
}
