// Chunked varlen prefill of the gated delta rule on the 64-token chunk grid,
// with 5th-generation tensor cores (tcgen05.mma, accumulators in TMEM).
//
// Routes and grid: vLLM page "Enable batch-invariant mixed decode and prefill
// for Qwen GDN" (section "How": fresh prefill rows go through chunk prefill),
// "GatedDeltaNet Automatic Prefix Caching" (section "Purpose": optional
// per-chunk intermediate states as one flat stream) and "Enable GDN
// batch-invariant prefix caching" (section "Purpose": 64-token chunks on one
// grid shared with prefix-cache hits).
//
// Chunked form (UT / WY representation of the delta rule, Yang et al.,
// "Parallelizing Linear Transformers with the Delta Rule over Sequence
// Length", NeurIPS 2024, with the gating of Gated DeltaNet, ICLR 2025).
// For a chunk of C = 64 tokens entering with state S0 (d_k x d_v), local
// index t, G_t = sum_{s<=t} g_s, gamma_t = exp(G_t):
//
//     A_ts  = beta_t exp(G_t - G_s) k_t.k_s   (s < t),   T = (I + A)^-1
//     V'    = V - diag(gamma) K S0
//     U     = T diag(beta) V'                              (the rows u_t)
//     O     = scale [diag(gamma) Q S0 + P U],  P_ts = exp(G_t - G_s) q_t.k_s (s <= t)
//     S_C   = gamma_C S0 + Ktil^T U,           Ktil_t = exp(G_C - G_t) k_t
//
// Everything is computed transposed so that TMEM lane j is value column j:
//     D1 = S0^T [Q;K]^T   (M = d_v, N = 128 tokens, K = d_k)
//     D3 = V'^T (T'')^T   (T'' = T diag(beta); M = d_v, N = 64, K = 64)
//     D5 = gamma_C S0^T + U^T Ktil     (the fp32 state, accumulated in TMEM)
//     D6 = U^T P^T
// and the Gram [Q;K] K^T (M = 128 tokens, N = 64, K = d_k) sits in its own
// TMEM columns.  Every tensor-core operand is fp16 (inputs convert exactly
// from bf16 except below 2^-14), accumulation and the state carry are fp32.
//
// One CTA (4 warps; thread j owns TMEM lane j) runs one (sequence, value
// head) chain through its chunks in order.  A chunk's arithmetic depends only
// on its own inputs and the fp32 state entering it, so results do not depend
// on the batch, and restarting from an emitted state reproduces the
// uninterrupted run bit for bit.
#include <cuda_fp16.h>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 128;
constexpr int kAS = 65;  // fp32 row stride of the 64x64 scratch matrices
// Upper bound on the wait for one group of MMAs, in SM clock cycles (~1 s):
// a wait that runs out reports GDN_DEV_TIMEOUT instead of hanging.
constexpr long long kWaitCycles = 2000000000LL;

template <int D>
struct Smem {
    // Tensor-core operand tiles (K-major, 128-byte swizzle, 1024-aligned).
    static constexpr uint32_t kQK = 0;                        // fp16 [128 rows: q then k][D]
    static constexpr uint32_t kS0T = kQK + 128 * D * 2;       // fp16 [128 rows j][D]  (S0^T)
    static constexpr uint32_t kVpT = kS0T + 128 * D * 2;      // fp16 [128 rows j][64] (V'^T); O staging
    static constexpr uint32_t kUT = kVpT + 128 * 64 * 2;      // fp16 [128 rows j][64] (U^T)
    static constexpr uint32_t kTpp = kUT + 128 * 64 * 2;      // fp16 [64 rows t][64]  (T diag(beta))
    static constexpr uint32_t kP = kTpp + 64 * 64 * 2;        // fp16 [64 rows t][64]  (P)
    static constexpr uint32_t kKtT = kP + 64 * 64 * 2;        // fp16 [D rows i][64]   (Ktil^T)
    // Plain buffers.
    static constexpr uint32_t kV = kKtT + D * 64 * 2;         // bf16 [64][D] values of the chunk
    static constexpr uint32_t kA = kV + 64 * D * 2;           // fp32 [64][kAS] strictly lower A
    static constexpr uint32_t kT = kA + 64 * kAS * 4;         // fp32 [64][kAS] T = (I + A)^-1
    static constexpr uint32_t kW = kT + 64 * kAS * 4;         // fp32 [3][16][16] inverse scratch
    static constexpr uint32_t kG = kW + 3 * 256 * 4;          // fp32 [64] cumulative log decay
    static constexpr uint32_t kGam = kG + 64 * 4;             // fp32 [64] exp(G_t)
    static constexpr uint32_t kDec = kGam + 64 * 4;           // fp32 [64] exp(G_C - G_t)
    static constexpr uint32_t kBeta = kDec + 64 * 4;          // fp32 [64]
    static constexpr uint32_t kGraw = kBeta + 64 * 4;         // fp32 [64] g of the chunk
    static constexpr uint32_t kBar = kGraw + 64 * 4;          // mbarrier (8 B)
    static constexpr uint32_t kTmem = kBar + 8;               // TMEM base address (4 B)
    static constexpr uint32_t kFlag = kTmem + 4;              // int (4 B)
    static constexpr uint32_t kEoff = kFlag + 4;              // long long [4] block reduction
    static constexpr uint32_t kBytes = kEoff + 32;
    static constexpr uint32_t kAlloc = kBytes + 1024;         // + alignment slack
};

// TMEM column map (512 columns allocated; lane j = value column j).
constexpr uint32_t kColD1 = 0;     // [0,64): (Q S0)^T, [64,128): (K S0)^T
constexpr uint32_t kColD3 = 128;   // U^T (fp32)
constexpr uint32_t kColD6 = 192;   // (P U)^T
constexpr uint32_t kColD5 = 256;   // S^T state, D columns
constexpr uint32_t kColGram = 384; // lanes 0..63: Q K^T rows, 64..127: K K^T rows
constexpr uint32_t kTmemCols = 512;

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// 8 bf16 (one uint4) -> 8 fp16 (one uint4), exact except below 2^-14.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 w) {
    uint4 r;
    r.x = pack_half2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u));
    r.y = pack_half2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
    r.z = pack_half2(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xffff0000u));
    r.w = pack_half2(__uint_as_float(w.w << 16), __uint_as_float(w.w & 0xffff0000u));
    return r;
}

__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
    return __half2float(*reinterpret_cast<__half *>(&h));
}

// Writes 64 fp32 values (scaled) as one fp16 row of a 64-wide K-major tile.
__device__ __forceinline__ void store_row64_f16(uint8_t *tile, uint32_t rows, uint32_t r, const float *x,
                                                int32_t *st = nullptr) {
    (void)st;
    if (!GDN_GUARD(st, r < rows && tc::sw128_chunk_offset(r, 7, rows) + 16 <= rows * 128u, 31, r)) return;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint4 v;
        v.x = pack_half2(x[8 * c + 0], x[8 * c + 1]);
        v.y = pack_half2(x[8 * c + 2], x[8 * c + 3]);
        v.z = pack_half2(x[8 * c + 4], x[8 * c + 5]);
        v.w = pack_half2(x[8 * c + 6], x[8 * c + 7]);
        *reinterpret_cast<uint4 *>(tile + tc::sw128_chunk_offset(r, c, rows)) = v;
    }
}

// Writes columns [c0, c0 + 32) of row r (fp32 bit patterns) as fp16 into a
// 128-row K-major SW128 tile.
__device__ __forceinline__ void store_f16_chunks32(uint8_t *tile, uint32_t r, int c0, const uint32_t (&x)[32]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 v;
        v.x = pack_half2(__uint_as_float(x[8 * q + 0]), __uint_as_float(x[8 * q + 1]));
        v.y = pack_half2(__uint_as_float(x[8 * q + 2]), __uint_as_float(x[8 * q + 3]));
        v.z = pack_half2(__uint_as_float(x[8 * q + 4]), __uint_as_float(x[8 * q + 5]));
        v.w = pack_half2(__uint_as_float(x[8 * q + 6]), __uint_as_float(x[8 * q + 7]));
        *reinterpret_cast<uint4 *>(tile + tc::sw128_chunk_offset(r, c0 / 8 + q, 128)) = v;
    }
}

__device__ __forceinline__ uint32_t lane_addr(uint32_t tbase, int warp, uint32_t col) {
    return tbase + (static_cast<uint32_t>(warp * 32) << 16) + col;
}

// Loads `n` (multiple of 32) consecutive fp32 TMEM columns of this thread's lane.
template <int N>
__device__ __forceinline__ void tmem_load_row(uint32_t taddr, float (&x)[N]) {
    static_assert(N % 32 == 0, "");
#ifdef GDN_DEBUG_CHECKS
    if ((taddr & 0xffffu) + N > kTmemCols) {
#pragma unroll
        for (int i = 0; i < N; ++i) x[i] = 0.f;
        return;
    }
#endif
#pragma unroll
    for (int c = 0; c < N; c += 32) {
        uint32_t r[32];
        tc::tmem_ld32(taddr + c, r);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[c + i] = __uint_as_float(r[i]);
    }
}

// Sum over s' < s of floor(L_s' / (64 E)), by the whole block.
__device__ int64_t emit_offset(const int32_t *cu, int s, int E, long long *part) {
    long long acc = 0;
    for (int i = threadIdx.x; i < s; i += blockDim.x) acc += (cu[i + 1] - cu[i]) / (kChunk * E);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
    __syncthreads();
    long long tot = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) tot += part[w];
    __syncthreads();
    return tot;
}

// T = (I + A)^-1 for a 64x64 strictly lower-triangular A (fp32, row stride
// kAS): the four 16x16 diagonal blocks by column forward substitution, then
// the block diagonals below, T_ab = -T_aa sum_{b<=m<a} A_am T_mb.  Only the
// lower block triangle of T is written.
__device__ void invert_unit_lower_64(const float *A, float *T, float *W, int tid) {
    if (tid < 64) {
        // Indices are masked so that every address stays inside the 64x64
        // matrices for any thread, whatever the compiler does with the branch.
        const int b = (tid >> 4) & 3, c = tid & 15, base = b * 16;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = (i == c) ? 1.f : 0.f;
#pragma unroll
        for (int i = 1; i < 16; ++i) {
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < i; ++j) acc = fmaf(A[(base + i) * kAS + base + j], x[j], acc);
            if (i > c) x[i] = -acc;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) T[(base + i) * kAS + base + c] = x[i];
    }
    __syncthreads();
    for (int lev = 1; lev < 4; ++lev) {
        const int nblk = 4 - lev;
        for (int e = tid; e < nblk * 256; e += kThreads) {
            const int b = e >> 8, i = (e >> 4) & 15, c = e & 15, a = b + lev;
            float acc = 0.f;
            for (int m = b; m < a; ++m)
#pragma unroll
                for (int kk = 0; kk < 16; ++kk)
                    acc = fmaf(A[(a * 16 + i) * kAS + m * 16 + kk], T[(m * 16 + kk) * kAS + b * 16 + c], acc);
            W[b * 256 + i * 16 + c] = acc;
        }
        __syncthreads();
        for (int e = tid; e < nblk * 256; e += kThreads) {
            const int b = e >> 8, i = (e >> 4) & 15, c = e & 15, a = b + lev;
            float acc = 0.f;
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
                acc = fmaf(T[(a * 16 + i) * kAS + a * 16 + kk], W[b * 256 + kk * 16 + c], acc);
            T[(a * 16 + i) * kAS + b * 16 + c] = -acc;
        }
        __syncthreads();
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_chunk_tc_kernel(const PrefillArgs a) {
    using L = Smem<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQK = sm + L::kQK, *sS0T = sm + L::kS0T, *sVpT = sm + L::kVpT, *sUT = sm + L::kUT;
    uint8_t *sTpp = sm + L::kTpp, *sP = sm + L::kP, *sKtT = sm + L::kKtT;
    uint16_t *sV = reinterpret_cast<uint16_t *>(sm + L::kV);
    float *sA = reinterpret_cast<float *>(sm + L::kA), *sT = reinterpret_cast<float *>(sm + L::kT);
    float *sW = reinterpret_cast<float *>(sm + L::kW), *sG = reinterpret_cast<float *>(sm + L::kG);
    float *sGam = reinterpret_cast<float *>(sm + L::kGam), *sDec = reinterpret_cast<float *>(sm + L::kDec);
    float *sBeta = reinterpret_cast<float *>(sm + L::kBeta), *sGraw = reinterpret_cast<float *>(sm + L::kGraw);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::kBar);
    uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(sm + L::kTmem);
    int *flag = reinterpret_cast<int *>(sm + L::kFlag);
    long long *part = reinterpret_cast<long long *>(sm + L::kEoff);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int seq = blockIdx.x / a.h_v, h = blockIdx.x % a.h_v;
    const int kh = h / (a.h_v / a.h_k);
    const int t0 = a.cu_seqlens[seq];
    const int Lseq = a.cu_seqlens[seq + 1] - t0;
    const int E = a.emit_every_chunks;
    const int64_t eoff = (E > 0 && a.chunk_states) ? emit_offset(a.cu_seqlens, seq, E, part) : 0;
    const int src = a.src_slot ? a.src_slot[seq] : -1;
    const int dst = a.dst_slot ? a.dst_slot[seq] : -1;
    const size_t ldq = static_cast<size_t>(a.h_k) * D, ldv = static_cast<size_t>(a.h_v) * D;

    if (src >= a.num_slots || dst >= a.num_slots) {
        if (tid == 0) report(a.dev_status, GDN_DEV_BAD_SLOT);
        for (int64_t e = tid; e < static_cast<int64_t>(Lseq) * (D / 8); e += kThreads) {
            const int64_t t = e / (D / 8), c = e % (D / 8);
            *reinterpret_cast<uint4 *>(a.o + (t0 + t) * ldv + static_cast<size_t>(h) * D + c * 8) =
                make_uint4(0, 0, 0, 0);
        }
        return;
    }

    // ---- set-up: TMEM, barrier, initial state ----------------------------------
    if (warp == 0) {
        tc::tmem_alloc(tmem_ptr, kTmemCols);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        tc::mbar_init(bar, 1);
        *flag = 0;
    }
    // Rows >= D of the transposed operand tiles stay zero (d = 64 pads M to 128).
    if (D < 128) {
        for (int e = tid; e < 128 * D * 2 / 16; e += kThreads)
            reinterpret_cast<uint4 *>(sS0T)[e] = make_uint4(0, 0, 0, 0);
        for (int e = tid; e < 128 * 64 * 2 / 16; e += kThreads) {
            reinterpret_cast<uint4 *>(sVpT)[e] = make_uint4(0, 0, 0, 0);
            reinterpret_cast<uint4 *>(sUT)[e] = make_uint4(0, 0, 0, 0);
        }
    }
    // Strict upper triangles of the scratch matrices stay zero.
    for (int e = tid; e < 64 * kAS; e += kThreads) {
        sA[e] = 0.f;
        sT[e] = 0.f;
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = *tmem_ptr;
    const uint32_t my_lane = lane_addr(tbase, warp, 0);
    (void)GDN_GUARD(a.dev_status, tbase == 0, 50, tbase);
    (void)GDN_GUARD(a.dev_status, (tc::smem_u32(sm) & 1023u) == 0 && tc::smem_u32(sm) + L::kBytes <= 232448u, 51,
                    tc::smem_u32(sm));
    const int j = tid;  // value column owned by this thread (valid when j < D)

    // Initial state S0^T row j: fp32 into TMEM (D5), fp16 into the S0^T
    // operand tile; or, for an empty sequence, straight to the destination.
    if (j < D) {
        const float *sp = (src >= 0 && GDN_GUARD(a.dev_status, src < a.num_slots, 3, src))
                              ? a.state + ((static_cast<size_t>(src) * a.h_v + h) * D + j) * D
                              : nullptr;
        float *dp = (Lseq == 0 && dst >= 0 && GDN_GUARD(a.dev_status, dst < a.num_slots, 4, dst))
                        ? a.state + ((static_cast<size_t>(dst) * a.h_v + h) * D + j) * D
                        : nullptr;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t r[32];
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (sp) v = __ldcg(reinterpret_cast<const float4 *>(sp + c0 + i));
                r[i] = __float_as_uint(v.x);
                r[i + 1] = __float_as_uint(v.y);
                r[i + 2] = __float_as_uint(v.z);
                r[i + 3] = __float_as_uint(v.w);
                if (dp) __stcg(reinterpret_cast<float4 *>(dp + c0 + i), v);
            }
            if (Lseq > 0) {
                tc::tmem_st32(my_lane + kColD5 + c0, r);
                store_f16_chunks32(sS0T, j, c0, r);
            }
        }
    }

    const uint32_t aQK = tc::smem_u32(sQK), aS0T = tc::smem_u32(sS0T), aVpT = tc::smem_u32(sVpT);
    const uint32_t aUT = tc::smem_u32(sUT), aTpp = tc::smem_u32(sTpp), aP = tc::smem_u32(sP);
    const uint32_t aKtT = tc::smem_u32(sKtT);
    uint32_t phase = 0;
    const int n_chunks = (Lseq + kChunk - 1) / kChunk;
    bool failed = false;

    // Issues nothing itself; every thread waits for the last commit.
    auto wait_mma = [&]() -> bool {
        const long long start = clock64();
        bool ok = false;
        while (!(ok = tc::mbar_try_wait(bar, phase)))
            if (clock64() - start > kWaitCycles) break;
        phase ^= 1u;
        tc::fence_after_sync();
        return __syncthreads_or(!ok) == 0;
    };

    for (int c = 0; c < n_chunks && !failed; ++c) {
        const int tok0 = t0 + c * kChunk;
        const int n = min(kChunk, Lseq - c * kChunk);

        // ---- L: chunk inputs -> smem (q, k as fp16 operand tiles; v as bf16) ----
        for (int e = tid; e < 64 * (D / 8); e += kThreads) {
            const int r = e / (D / 8), cc = e % (D / 8);
            uint4 qv = make_uint4(0, 0, 0, 0), kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
            if (r < n && GDN_GUARD(a.dev_status, tok0 + r < a.total_tokens, 1, tok0 + r)) {
                const size_t row = static_cast<size_t>(tok0 + min(r, n - 1));  // always a row of this chunk
                qv = bf16x8_to_f16x8(__ldg(reinterpret_cast<const uint4 *>(a.q + row * ldq + kh * D + cc * 8)));
                kv = bf16x8_to_f16x8(__ldg(reinterpret_cast<const uint4 *>(a.k + row * ldq + kh * D + cc * 8)));
                vv = __ldg(reinterpret_cast<const uint4 *>(a.v + row * ldv + static_cast<size_t>(h) * D + cc * 8));
            }
            if (!GDN_GUARD(a.dev_status, tc::sw128_chunk_offset(64 + r, cc, 128) + 16 <= 128u * D * 2 &&
                                            r * D + cc * 8 + 8 <= 64 * D, 11, e))
                continue;
            *reinterpret_cast<uint4 *>(sQK + tc::sw128_chunk_offset(r, cc, 128)) = qv;
            *reinterpret_cast<uint4 *>(sQK + tc::sw128_chunk_offset(64 + r, cc, 128)) = kv;
            *reinterpret_cast<uint4 *>(sV + r * D + cc * 8) = vv;
        }
        if (tid < 64) {
            const size_t gi = static_cast<size_t>(tok0 + min(tid, n - 1)) * a.h_v + h;
            const bool in = tid < n && GDN_GUARD(a.dev_status, tok0 + tid < a.total_tokens, 2, tok0 + tid);
            sGraw[tid] = in ? a.g[gi] : 0.f;
            sBeta[tid] = in ? a.beta[gi] : 0.f;
        }
        __syncthreads();
        if (warp == 0) {
            // inclusive prefix sum of g over the chunk, fixed order
            const int l = tid;
            const float g0 = sGraw[2 * l], g1 = sGraw[2 * l + 1];
            const float pair = g0 + g1;
            float incl = pair;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, o);
                if (l >= o) incl += y;
            }
            const float excl = incl - pair;
            sG[2 * l] = excl + g0;
            sG[2 * l + 1] = excl + g0 + g1;
        }
        __syncwarp();
        __syncthreads();
        if (tid < 64) {
            sGam[tid] = expf(sG[tid]);
            sDec[tid] = expf(sG[63] - sG[tid]);
        }
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();

        // ---- M1: Gram [Q;K] K^T and D1 = S0^T [Q;K]^T ----------------------------
        if (tid == 0) {
            tc::fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * 128 * 128 + (kk & 3) * 32;
                tc::mma_f16(tbase + kColGram, tc::desc_k_sw128(aQK + off), tc::desc_k_sw128(aQK + off + 64 * 128),
                            tc::idesc_f16_f32acc(128, 64), kk > 0);
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * 128 * 128 + (kk & 3) * 32;
                tc::mma_f16(tbase + kColD1, tc::desc_k_sw128(aS0T + off), tc::desc_k_sw128(aQK + off),
                            tc::idesc_f16_f32acc(128, 128), kk > 0);
            }
            tc::mma_commit(bar);
        }
        __syncwarp();
        if (!wait_mma()) {
            failed = true;
            break;
        }

        // ---- G: P (from Q K^T rows) and A (from K K^T rows) ------------------------
        {
            float x[64];
            tmem_load_row<64>(my_lane + kColGram, x);
            if (tid < 64) {
                const int t = tid & 63;
                const float Gt = sG[t];
#pragma unroll
                for (int s = 0; s < 64; ++s) x[s] = (s <= t) ? expf(Gt - sG[s]) * x[s] : 0.f;
                store_row64_f16(sP, 64, t, x, a.dev_status);
            } else {
                const int i = tid & 63;
                const float Gi = sG[i], bi = sBeta[i];
#pragma unroll
                for (int s = 0; s < 64; ++s)
                    if (s < i && GDN_GUARD(a.dev_status, i * kAS + s < 64 * kAS, 15, i)) sA[i * kAS + s] = bi * (expf(Gi - sG[s]) * x[s]);
            }
        }
        // Ktil^T[i][t] = exp(G_C - G_t) k_t[i]
        if (tid < D) {
            const int i = tid & (D - 1);
            float x[64];
#pragma unroll
            for (int t = 0; t < 64; ++t) {
                const uint16_t kb = *reinterpret_cast<const uint16_t *>(sQK + tc::sw128_offset(64 + t, i, 128));
                x[t] = sDec[t] * half_bits_to_float(kb);
            }
            store_row64_f16(sKtT, D, i, x, a.dev_status);
        }
        __syncthreads();

        // ---- I: T = (I + A)^-1, T'' = T diag(beta) ----------------------------------
        invert_unit_lower_64(sA, sT, sW, tid);
        if (tid < 64) {
            // Row index masked: the loads stay inside T even if they are
            // executed for threads outside the branch.
            const int t = tid & 63;
            float x[64];
#pragma unroll
            for (int s = 0; s < 64; ++s) x[s] = (s <= t) ? sT[t * kAS + s] * sBeta[s] : 0.f;
            store_row64_f16(sTpp, 64, t, x, a.dev_status);
        }

        // ---- C2: V'^T = V^T - (K S0)^T diag(gamma); gamma_C scales the state -----
        if (j < D) {
            float ks[64];
            tmem_load_row<64>(my_lane + kColD1 + 64, ks);
#pragma unroll
            for (int t = 0; t < 64; ++t) {
                const uint16_t vb = sV[t * D + (j & (D - 1))];
                ks[t] = __uint_as_float(static_cast<uint32_t>(vb) << 16) - sGam[t] * ks[t];
            }
            store_row64_f16(sVpT, 128, j, ks, a.dev_status);
        }
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                tc::mma_f16(tbase + kColD3, tc::desc_k_sw128(aVpT + kk * 32), tc::desc_k_sw128(aTpp + kk * 32),
                            tc::idesc_f16_f32acc(128, 64), kk > 0);
            tc::mma_commit(bar);
        }
        __syncwarp();
        if (j < D) {
            const float gC = sGam[63];
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t r[32];
                tc::tmem_ld32(my_lane + kColD5 + c0, r);
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(gC * __uint_as_float(r[i]));
                tc::tmem_st32(my_lane + kColD5 + c0, r);
            }
        }
        tc::fence_before_sync();
        if (!wait_mma()) {
            failed = true;
            break;
        }

        // ---- C4: U^T to fp16; D5 += U^T Ktil, D6 = U^T P^T ---------------------------
        if (j < D) {
            float u[64];
            tmem_load_row<64>(my_lane + kColD3, u);
            store_row64_f16(sUT, 128, j, u, a.dev_status);
        }
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                tc::mma_f16(tbase + kColD5, tc::desc_k_sw128(aUT + kk * 32), tc::desc_k_sw128(aKtT + kk * 32),
                            tc::idesc_f16_f32acc(128, D), 1);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                tc::mma_f16(tbase + kColD6, tc::desc_k_sw128(aUT + kk * 32), tc::desc_k_sw128(aP + kk * 32),
                            tc::idesc_f16_f32acc(128, 64), kk > 0);
            tc::mma_commit(bar);
        }
        __syncwarp();
        if (!wait_mma()) {
            failed = true;
            break;
        }

        // ---- C6: new state, emission, outputs -----------------------------------------
        uint16_t *sO = reinterpret_cast<uint16_t *>(sVpT);  // V'^T is consumed: reuse as O staging
        if (j < D) {
            const bool emit = E > 0 && a.chunk_states && n == kChunk && ((c + 1) % E) == 0;
            float *ep = nullptr;
            if (emit) {
                const int64_t idx = eoff + (c + 1) / E - 1;
                if (GDN_GUARD(a.dev_status, idx >= 0 && idx < a.chunk_capacity, 5, idx))
                    ep = a.chunk_states + ((static_cast<size_t>(idx) * a.h_v + h) * D + j) * D;
            }
            float *dp = (c == n_chunks - 1 && dst >= 0 && GDN_GUARD(a.dev_status, dst < a.num_slots, 4, dst))
                            ? a.state + ((static_cast<size_t>(dst) * a.h_v + h) * D + j) * D
                            : nullptr;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t r[32];
                tc::tmem_ld32(my_lane + kColD5 + c0, r);
                store_f16_chunks32(sS0T, j, c0, r);
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const float4 v = make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]),
                                                 __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
                    if (ep) __stcg(reinterpret_cast<float4 *>(ep + c0 + i), v);
                    if (dp) __stcg(reinterpret_cast<float4 *>(dp + c0 + i), v);
                }
            }
            float qs[64], pu[64];
            tmem_load_row<64>(my_lane + kColD1, qs);
            tmem_load_row<64>(my_lane + kColD6, pu);
#pragma unroll
            for (int t = 0; t < 64; ++t) {
                const float ov = a.scale * fmaf(sGam[t], qs[t], pu[t]);
                if (GDN_GUARD(a.dev_status, t * D + j < 64 * 128, 17, t * D + j)) sO[t * D + j] = float_to_bf16_bits(ov);
            }
        }
        tc::fence_before_sync();
        __syncthreads();
        for (int e = tid; e < n * (D / 8); e += kThreads) {
            const int t = e / (D / 8), cc = e % (D / 8);
            if (!GDN_GUARD(a.dev_status, tok0 + t < a.total_tokens, 6, tok0 + t)) continue;
            *reinterpret_cast<uint4 *>(a.o + static_cast<size_t>(tok0 + t) * ldv + static_cast<size_t>(h) * D +
                                       cc * 8) = *reinterpret_cast<const uint4 *>(sO + t * D + cc * 8);
        }
        __syncthreads();
    }

    if (failed) {
        if (tid == 0) report(a.dev_status, GDN_DEV_TIMEOUT);
        // Give MMAs that may still be in flight a bounded time to finish
        // before the TMEM they write is released.
        const long long start = clock64();
        while (!tc::mbar_try_wait(bar, phase) && clock64() - start < kWaitCycles) {
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tbase, kTmemCols);
}

template <int D>
cudaError_t launch_d(const PrefillArgs &a, cudaStream_t stream) {
    const uint32_t smem = Smem<D>::kAlloc;
    cudaError_t e = cudaFuncSetAttribute(prefill_chunk_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    prefill_chunk_tc_kernel<D><<<a.num_seqs * a.h_v, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, int d, int64_t total_tokens, int32_t max_seqlen,
                           cudaStream_t stream) {
    (void)total_tokens;
    (void)max_seqlen;
    if (a.num_seqs == 0) return cudaSuccess;
    return d == 128 ? launch_d<128>(a, stream) : launch_d<64>(a, stream);
}

}  // namespace gdn
