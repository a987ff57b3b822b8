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
// Products are computed transposed so that TMEM lane j is value column j:
//     D1 = S0^T [Q;K]^T  (M = d_v, N = 128 tokens, K = d_k), double-buffered
//     D3 = V'^T T''^T    (T'' = T diag(beta); reuses the K half of D1)
//     D5 = gamma_C S0^T + (diag(dec) U)^T K,  dec_t = exp(G_C - G_t)
//          (the fp32 state, accumulated in TMEM; K is read MN-major straight
//          from its TMA tile, so Ktil is never formed)
//     D6 = U^T P^T
// and the Gram [Q;K] K^T (M = 128 tokens, N = 64, K = d_k).  Operands are
// fp16 (inputs convert exactly from bf16 except below 2^-14); accumulation
// and the state carry are fp32.
//
// One CTA runs one (sequence, value head) chain, warp-specialised:
//   chain group (warps 0-7; warps w and w + 4 share TMEM lane quarter w, so
//     lane j is served by two threads, each taking half of the row's tokens
//     or state columns): the steps that depend on the state,
//     S1 -> V' -> S3 -> U -> S5/S6 -> new state, plus the output of the
//     previous chunk while S1 runs;
//   prep group (warps 8-15, lanes split the same way): the chunk-local
//     operands of the next chunk -- Q/K tiles (TMA into a ring of three
//     slots, issued a whole chunk ahead and converted to fp16 in place
//     while the previous chunk's diagonal blocks are solved), decays, Gram,
//     P, A, T = (I + A)^-1 (diagonal 16x16 blocks by substitution, then two
//     doubling levels) and T'' -- into a double-buffered stage, handed over
//     through mbarriers.
// A chunk's arithmetic depends only on its own inputs and the fp32 state
// entering it, so results do not depend on the batch, and restarting from an
// emitted state reproduces the uninterrupted run bit for bit.
//
// Every shared-memory index that depends on the thread index is masked to
// its array's range, so no address can leave the allocation even for a
// thread outside the branch that guards it.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 512;  // chain group + prep group
constexpr int kGroup = 256;    // 8 warps per group: two warps per TMEM lane quarter
constexpr int kBarChain = 1;   // named barrier ids (0 is __syncthreads)
constexpr int kBarPrep = 2;
// Upper bound on every wait, in SM clock cycles (~1 s): a wait that runs out
// reports GDN_DEV_TIMEOUT instead of hanging.
constexpr long long kWaitCycles = 2000000000LL;
constexpr int kMaxOrder = 2048;

struct PrefillLaunch {
    CUtensorMap tm_q, tm_k;  // q, k as 2-D [T][h_k d] bf16, 64 x 64 boxes, 128-byte swizzle
    PrefillArgs a;
    int32_t n_order;
    int32_t order[kMaxOrder];  // launch rank -> sequence, longest first
};

template <int D>
struct Smem {
    // Tensor-core operand tiles (K-major, 128-byte swizzle, 1024-aligned).
    static constexpr uint32_t kQKBytes = 128 * D * 2;          // fp16 [128 rows: q then k][D]
    static constexpr uint32_t kQK0 = 0;                          // ring of three slots
    static constexpr uint32_t kTpp0 = kQK0 + 3 * kQKBytes;     // fp16 [64 rows t][64]  T''
    static constexpr uint32_t kTpp1 = kTpp0 + 8192;
    static constexpr uint32_t kP0 = kTpp1 + 8192;              // fp16 [64 rows t][64]  P
    static constexpr uint32_t kP1 = kP0 + 8192;
    static constexpr uint32_t kS0T = kP1 + 8192;               // fp16 [128 rows j][D]  S0^T
    static constexpr uint32_t kVpT = kS0T + 128 * D * 2;       // fp16 [128 rows j][64] V'^T, then (diag(dec) U)^T
    static constexpr uint32_t kUT = kVpT + 16384;              // fp16 [128 rows j][64] U^T
    // Plain buffers.
    static constexpr uint32_t kGam0 = kUT + 16384;             // f32 [64] exp(G_t), stage 0
    static constexpr uint32_t kGam1 = kGam0 + 256;
    static constexpr uint32_t kGamC = kGam1 + 256;             // f32 [2][64] chain group's copies
    static constexpr uint32_t kM = kGamC + 512;                // f32 [64][kLdM] A, then T
    static constexpr uint32_t kW = kM + 64 * 68 * 4;           // f32 [4][16][16] block products
    static constexpr uint32_t kG = kW + 4096;                  // f32 [64] cumulative log decay
    static constexpr uint32_t kBeta = kG + 256;                // f32 [64]
    static constexpr uint32_t kGraw = kBeta + 256;             // f32 [64]
    static constexpr uint32_t kDec = kGraw + 256;              // f32 [2][64] exp(G_C - G_t), per stage
    static constexpr uint32_t kBars = kDec + 512;              // 9 mbarriers
    static constexpr uint32_t kTmem = kBars + 128;             // TMEM base address
    static constexpr uint32_t kFail = kTmem + 4;               // int
    static constexpr uint32_t kEoff = kFail + 4;               // long long [16]
    static constexpr uint32_t kBytes = kEoff + 128;
    static constexpr uint32_t kAlloc = kBytes + 1024;          // + alignment slack
    static_assert(kS0T % 1024 == 0 && kVpT % 1024 == 0 && kUT % 1024 == 0 && kBars % 8 == 0, "");
    static_assert(kTpp0 % 1024 == 0 && kP0 % 1024 == 0 && kQKBytes % 1024 == 0, "");
    static_assert(kM % 16 == 0 && kW % 16 == 0, "float4 access to the scratch");
    static_assert(kAlloc <= 232448, "shared memory budget");
};

// TMEM column map (512 columns; lane j = value column j).
constexpr uint32_t kColD1 = 0;      // two buffers of 128: [0,64) (Q S0)^T, [64,128) (K S0)^T then U^T
constexpr uint32_t kColD5 = 256;    // S^T state, D columns
constexpr uint32_t kColD6 = 384;    // (P U)^T
constexpr uint32_t kColGram = 448;  // lanes 0..63: Q K^T rows, 64..127: K K^T rows
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

// TMA: one 2-D box of a tensor map into shared memory, completing on an
// mbarrier that expects the box's bytes.
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            tc::smem_u32(smem_dst)),
        "l"(map), "r"(x), "r"(y), "r"(tc::smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc::smem_u32(bar)), "r"(bytes)
                 : "memory");
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

// Writes 8 fp32 values as the 16-byte fp16 chunk `chunk` of row r of a K-major
// SW128 tile of `rows` rows.
__device__ __forceinline__ void store_chunk8_f16(uint8_t *tile, uint32_t rows, uint32_t r, uint32_t chunk,
                                                 const float *x) {
    uint4 v;
    v.x = pack_half2(x[0], x[1]);
    v.y = pack_half2(x[2], x[3]);
    v.z = pack_half2(x[4], x[5]);
    v.w = pack_half2(x[6], x[7]);
    *reinterpret_cast<uint4 *>(tile + tc::sw128_chunk_offset(r, chunk, rows)) = v;
}

__device__ __forceinline__ uint32_t lane_addr(uint32_t tbase, int warp, uint32_t col) {
    return tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16) + col;
}

template <int N>
__device__ __forceinline__ void tmem_load_row(uint32_t taddr, float (&x)[N]) {
    static_assert(N % 32 == 0, "");
#pragma unroll
    for (int c = 0; c < N; c += 32) {
        uint32_t r[32];
        tc::tmem_ld32(taddr + c, r);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[c + i] = __uint_as_float(r[i]);
    }
}

// Group barrier (named barrier over the group's 256 threads).
__device__ __forceinline__ void group_sync(int id) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(kGroup) : "memory");
}

// Group barrier that returns true if any thread of the group passed `pred`.
__device__ __forceinline__ bool group_any(int id, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(kGroup)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}

// Bounded wait for the phase of `bar` with the given parity.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    const long long start = clock64();
    while (!tc::mbar_try_wait(bar, parity))
        if (clock64() - start > kWaitCycles) return false;
    return true;
}

// Row stride of the 64x64 fp32 scratch: 68 floats keep 16-byte alignment and
// put 8 consecutive rows on disjoint bank quads.
constexpr int kLdM = 68;

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

// In place, M := (I + M)^-1 for a 64x64 strictly lower-triangular M (the
// diagonal and upper triangle of M are ignored; the result has unit diagonal
// and zeros above it inside the diagonal blocks), in two parts run by the
// prep group (p = thread index within the group, 0..255).
//
// Part 1 (threads p < 64, block b = p / 16, column c = p % 16): the four
// 16x16 diagonal blocks by right-looking forward substitution; each step
// finishes x_j and updates the later rows independently of each other.
// The new columns are kept in x[] and written by invert_diag_store after a
// group barrier, once every thread has read the block's A entries.
__device__ __forceinline__ void invert_diag_solve(const float *M, int p, float (&x)[16]) {
    const int c = p & 15, base = ((p >> 4) & 3) * 16;
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const float xj = (j < c) ? 0.f : (j == c ? 1.f : -acc[j]);
        x[j] = xj;
#pragma unroll
        for (int i = j + 1; i < 16; ++i) acc[i] = fmaf(M[(base + i) * kLdM + base + j], xj, acc[i]);
    }
}

// Also writes the block's columns of T'' = T diag(beta) as fp16 into the
// 64-row K-major operand tile Tpp (upper blocks of Tpp stay zero).
__device__ __forceinline__ void invert_diag_store(float *M, int p, const float (&x)[16], uint8_t *Tpp,
                                                  const float *beta) {
    const int c = p & 15, base = ((p >> 4) & 3) * 16;
    const float bc = beta[base + c];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        M[(base + i) * kLdM + base + c] = x[i];
        *reinterpret_cast<__half *>(Tpp + tc::sw128_offset(base + i, base + c, 64)) = __float2half_rn(x[i] * bc);
    }
}

__device__ __forceinline__ void fma4(float4 &acc, float a, const float4 &t) {
    acc.x = fmaf(a, t.x, acc.x);
    acc.y = fmaf(a, t.y, acc.y);
    acc.z = fmaf(a, t.z, acc.z);
    acc.w = fmaf(a, t.w, acc.w);
}

// Part 2, the off-diagonal blocks, as two doubling levels (16 block
// products in four phases): with T_aa the inverted diagonal
// blocks,
//   level 1 (pairs of 16-blocks):  T_10 = -T_11 (A_10 T_00),  T_32 = -T_33 (A_32 T_22);
//   level 2 (rows 32..63 x columns 0..31):  X = A_B T_top,  T_B = -T_bottom X,
//   T_top = [[T_00, 0], [T_10, T_11]],  T_bottom = [[T_22, 0], [T_32, T_33]],
//   i.e. X_a0 = A_a0 T_00 + A_a1 T_10, X_a1 = A_a1 T_11 (a = 2, 3),
//        T_2b = -T_22 X_2b,  T_3b = -(T_32 X_2b + T_33 X_3b).
// Level 1 runs in the two warps that solved the diagonal blocks (warp
// barriers only); each level-2 output 16x16 block is computed by 64 threads
// (row i = (p/4) % 16, columns 4 (p%4) .. + 3, float4 accesses) with
// compile-time block indices per task.  Results go to M and, scaled by beta, as fp16 to the
// T'' tile.  The caller provides the barrier after the last phase.
template <int LDX, int LDY>
__device__ __forceinline__ void block_mac(float4 &acc, const float *X, const float *Y, int i, int cq) {
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
        const float4 x4 = *reinterpret_cast<const float4 *>(X + i * LDX + 4 * k4);
        const float *y = Y + (4 * k4) * LDY + 4 * cq;
        fma4(acc, x4.x, *reinterpret_cast<const float4 *>(y));
        fma4(acc, x4.y, *reinterpret_cast<const float4 *>(y + LDY));
        fma4(acc, x4.z, *reinterpret_cast<const float4 *>(y + 2 * LDY));
        fma4(acc, x4.w, *reinterpret_cast<const float4 *>(y + 3 * LDY));
    }
}

template <int A, int B>
__device__ __forceinline__ void store_t_block(float *M, uint8_t *Tpp, const float *beta, int i, int cq,
                                              const float4 &acc) {
    const int row = A * 16 + i, col = B * 16 + 4 * cq;
    *reinterpret_cast<float4 *>(M + row * kLdM + col) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
    const float4 b4 = *reinterpret_cast<const float4 *>(beta + col);
    uint2 hv;
    hv.x = pack_half2(-acc.x * b4.x, -acc.y * b4.y);
    hv.y = pack_half2(-acc.z * b4.z, -acc.w * b4.w);
    *reinterpret_cast<uint2 *>(Tpp + tc::sw128_offset(row, col, 64)) = hv;
}

#define GDN_MB(a, b) (M + ((a) * 16) * kLdM + (b) * 16)
// Level 1 by one warp (the warp that solved diagonal blocks A-1 and A):
// lane = (row i = lane / 2, columns 8 (lane % 2) .. + 7), two float4 each;
// Y_{A,A-1} = A_{A,A-1} T_{A-1,A-1} into W block (A == 3), then
// T_{A,A-1} = -T_AA Y, with warp barriers only.
template <int A>
__device__ __forceinline__ void level1_warp(float *M, float *W, int lane, uint8_t *Tpp, const float *beta) {
    const int i = (lane >> 1) & 15, h = lane & 1;
    float *Wy = W + (A == 3 ? 256 : 0);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        block_mac<kLdM, kLdM>(acc, M + (A * 16) * kLdM + (A - 1) * 16, M + ((A - 1) * 16) * kLdM + (A - 1) * 16, i,
                              2 * h + u);
        *reinterpret_cast<float4 *>(Wy + i * 16 + 4 * (2 * h + u)) = acc;
    }
    __syncwarp();
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        block_mac<kLdM, 16>(acc, M + (A * 16) * kLdM + A * 16, Wy, i, 2 * h + u);
        store_t_block<A, A - 1>(M, Tpp, beta, i, 2 * h + u, acc);
    }
}

template <int A, int B>  // level 2, X_AB into W block 2 (A - 2) + B
__device__ __forceinline__ void l2_x(float *M, float *W, int i, int cq) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (B == 0) block_mac<kLdM, kLdM>(acc, GDN_MB(A, 0), GDN_MB(0, 0), i, cq);
    block_mac<kLdM, kLdM>(acc, GDN_MB(A, 1), GDN_MB(1, B), i, cq);
    *reinterpret_cast<float4 *>(W + (2 * (A - 2) + B) * 256 + i * 16 + 4 * cq) = acc;
}
template <int A, int B>  // level 2, T_AB = -(T_A2 X_2B + [A == 3] T_33 X_3B)
__device__ __forceinline__ void l2_t(float *M, float *W, int i, int cq, uint8_t *Tpp, const float *beta) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    block_mac<kLdM, 16>(acc, GDN_MB(A, 2), W + B * 256, i, cq);
    if (A == 3) block_mac<kLdM, 16>(acc, GDN_MB(3, 3), W + (2 + B) * 256, i, cq);
    store_t_block<A, B>(M, Tpp, beta, i, cq, acc);
}
#undef GDN_MB

// Level 2 (level 1 was done per warp right after the diagonal blocks).
__device__ __forceinline__ void invert_offdiag(float *M, float *W, int p, uint8_t *Tpp, const float *beta) {
    const int task = (p >> 6) & 3, i = (p >> 2) & 15, cq = p & 3;  // task uniform over 2 warps
    switch (task) {
        case 0: l2_x<2, 0>(M, W, i, cq); break;
        case 1: l2_x<2, 1>(M, W, i, cq); break;
        case 2: l2_x<3, 0>(M, W, i, cq); break;
        default: l2_x<3, 1>(M, W, i, cq); break;
    }
    group_sync(kBarPrep);
    switch (task) {
        case 0: l2_t<2, 0>(M, W, i, cq, Tpp, beta); break;
        case 1: l2_t<2, 1>(M, W, i, cq, Tpp, beta); break;
        case 2: l2_t<3, 0>(M, W, i, cq, Tpp, beta); break;
        default: l2_t<3, 1>(M, W, i, cq, Tpp, beta); break;
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_chunk_tc_kernel(const __grid_constant__ PrefillLaunch L) {
    using SM = Smem<D>;
    const PrefillArgs &a = L.a;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // Stage s (chunk parity) buffers, by offset from stage 0.
    auto sQK = [&](int st) { return sm + SM::kQK0 + st * SM::kQKBytes; };
    auto sTpp = [&](int st) { return sm + SM::kTpp0 + st * 8192; };
    auto sP = [&](int st) { return sm + SM::kP0 + st * 8192; };
    auto sGam = [&](int st) { return reinterpret_cast<float *>(sm + SM::kGam0 + st * 256); };
    auto sGamC = [&](int st) { return reinterpret_cast<float *>(sm + SM::kGamC + st * 256); };
    uint8_t *sS0T = sm + SM::kS0T, *sVpT = sm + SM::kVpT, *sUT = sm + SM::kUT;
    float *sM = reinterpret_cast<float *>(sm + SM::kM), *sW = reinterpret_cast<float *>(sm + SM::kW);
    float *sG = reinterpret_cast<float *>(sm + SM::kG), *sBeta = reinterpret_cast<float *>(sm + SM::kBeta);
    float *sGraw = reinterpret_cast<float *>(sm + SM::kGraw);
    auto sDec = [&](int st) { return reinterpret_cast<float *>(sm + SM::kDec + st * 256); };
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + SM::kBars);
    // ready / freeb per stage (chunk parity); tma_bar per Q/K slot (chunk mod 3).
    uint64_t *mma_bar = bars + 0, *gram_bar = bars + 1, *ready = bars + 2, *freeb = bars + 4, *tma_bar = bars + 6;
    uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(sm + SM::kTmem);
    int *fail = reinterpret_cast<int *>(sm + SM::kFail);
    long long *part = reinterpret_cast<long long *>(sm + SM::kEoff);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int rank = blockIdx.x / a.h_v, h = blockIdx.x % a.h_v;
    const int seq = rank < L.n_order ? L.order[rank] : rank;
    const int kh = h / (a.h_v / a.h_k);
    const int t0 = a.cu_seqlens[seq];
    const int Lseq = a.cu_seqlens[seq + 1] - t0;
    const int E = a.emit_every_chunks;
    const int64_t eoff = (E > 0 && a.chunk_states) ? emit_offset(a.cu_seqlens, seq, E, part) : 0;
    const int emit_first = a.emit_table ? a.emit_first[seq] : 0;
    const int src = a.src_slot ? a.src_slot[seq] : -1;
    const int dst = a.dst_slot ? a.dst_slot[seq] : -1;
    const size_t ldq = static_cast<size_t>(a.h_k) * D, ldv = static_cast<size_t>(a.h_v) * D;
    const int n_chunks = (Lseq + kChunk - 1) / kChunk;

    if (src >= a.num_slots || dst >= a.num_slots) {
        if (tid == 0) report(a.dev_status, GDN_DEV_BAD_SLOT);
        for (int64_t e = tid; e < static_cast<int64_t>(Lseq) * (D / 8); e += kThreads) {
            const int64_t t = e / (D / 8), c = e % (D / 8);
            *reinterpret_cast<uint4 *>(a.o + (t0 + t) * ldv + static_cast<size_t>(h) * D + c * 8) =
                make_uint4(0, 0, 0, 0);
        }
        return;
    }

    // ---- set-up ----------------------------------------------------------------------
    if (warp == 0) {
        tc::tmem_alloc(tmem_ptr, kTmemCols);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        tc::mbar_init(mma_bar, 1);
        tc::mbar_init(gram_bar, 1);
        tc::mbar_init(ready + 0, kGroup);
        tc::mbar_init(ready + 1, kGroup);
        tc::mbar_init(freeb + 0, kGroup);
        tc::mbar_init(freeb + 1, kGroup);
        tc::mbar_init(tma_bar + 0, 1);
        tc::mbar_init(tma_bar + 1, 1);
        tc::mbar_init(tma_bar + 2, 1);
        *fail = 0;
    }
    for (int e = tid; e < 2 * 8192 / 16; e += kThreads)  // upper blocks of T'' stay zero
        reinterpret_cast<uint4 *>(sm + SM::kTpp0)[e] = make_uint4(0, 0, 0, 0);
    if (D < 128) {  // rows >= D of the transposed operand tiles stay zero (d = 64 pads M to 128)
        for (int e = tid; e < 128 * D * 2 / 16; e += kThreads)
            reinterpret_cast<uint4 *>(sS0T)[e] = make_uint4(0, 0, 0, 0);
        for (int e = tid; e < 16384 / 16; e += kThreads) {
            reinterpret_cast<uint4 *>(sVpT)[e] = make_uint4(0, 0, 0, 0);
            reinterpret_cast<uint4 *>(sUT)[e] = make_uint4(0, 0, 0, 0);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = *tmem_ptr;
    const uint32_t my_lane = lane_addr(tbase, warp, 0);

    if (warp < 8) {
        // ============================ chain group ==============================
        // Thread (j, hf): value column j (TMEM lane j), half hf of the row's work.
        const int j = tid & 127, hf = tid >> 7;
        const int jm = j & (D - 1);
        constexpr int kHalfD = D / 2;  // state columns per thread
        // Initial state row j, columns [hf D/2, (hf+1) D/2): fp32 into D5, fp16
        // into the S0^T tile; or, for an empty sequence, to the destination.
        if (j < D) {
            const float *sp = src >= 0 ? a.state + ((static_cast<size_t>(src) * a.h_v + h) * D + jm) * D : nullptr;
            float *dp = (Lseq == 0 && dst >= 0) ? a.state + ((static_cast<size_t>(dst) * a.h_v + h) * D + jm) * D
                                                : nullptr;
#pragma unroll 1
            for (int c0 = hf * kHalfD; c0 < (hf + 1) * kHalfD; c0 += 32) {
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
                    store_f16_chunks32(sS0T, jm, c0, r);
                }
            }
        }
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        group_sync(kBarChain);

        // Shared-memory descriptors; a K step adds its byte offset / 16.
        const uint64_t dS0T = tc::desc_k_sw128(tc::smem_u32(sS0T));
        const uint64_t dVpT = tc::desc_k_sw128(tc::smem_u32(sVpT));
        const uint64_t dUT = tc::desc_k_sw128(tc::smem_u32(sUT));
        constexpr uint32_t kIdN128 = tc::idesc_f16_f32acc(128, 128), kIdN64 = tc::idesc_f16_f32acc(128, 64);
        constexpr uint32_t kIdNDbmn = tc::idesc_f16_f32acc_bmn(128, D);  // B (the K tile) MN-major
        uint32_t mma_phase = 0;
        bool failed = false;
        int prev_n = 0, prev_tok0 = 0;
        uint16_t *sOst = reinterpret_cast<uint16_t *>(sVpT);
        uint16_t *sVst = reinterpret_cast<uint16_t *>(sUT);

        // Output of a finished chunk: o_t = scale (gamma_t (Q S0)_t + (P U)_t),
        // tokens t = 32 hf .. 32 hf + 31 per thread, staged as bf16 [t][D] in
        // the V'^T tile (free between S3 of that chunk and C2 of the next) and
        // stored with 16-byte writes.
        auto output = [&](int buf, int n_out, int tok_out) {
            if (j < D) {
                float qs[32], pu[32];
                tmem_load_row<32>(my_lane + kColD1 + 128 * buf + 32 * hf, qs);
                tmem_load_row<32>(my_lane + kColD6 + 32 * hf, pu);
                const float *gam = sGamC(buf) + 32 * hf;
#pragma unroll
                for (int i4 = 0; i4 < 32; i4 += 4) {
                    const float4 g4 = *reinterpret_cast<const float4 *>(gam + i4);
                    const float gg[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        sOst[(32 * hf + i4 + u) * D + jm] =
                            float_to_bf16_bits(a.scale * fmaf(gg[u], qs[i4 + u], pu[i4 + u]));
                }
            }
            tc::fence_before_sync();
            group_sync(kBarChain);
            for (int e = tid; e < n_out * (D / 8); e += kGroup) {
                const int t = e / (D / 8), cc = e % (D / 8);
                *reinterpret_cast<uint4 *>(a.o + static_cast<size_t>(tok_out + t) * ldv + static_cast<size_t>(h) * D +
                                           cc * 8) = *reinterpret_cast<const uint4 *>(sOst + t * D + cc * 8);
            }
            // the staging tile is next written by C2, after the S1 barrier
        };

        for (int c = 0; c < n_chunks; ++c) {
            const int s = c & 1, qs = c % 3;
            const int tok0 = t0 + c * kChunk;
            const int n = min(kChunk, Lseq - c * kChunk);
            const uint32_t d1 = tbase + kColD1 + 128 * s;
            const uint32_t d1_lane = my_lane + kColD1 + 128 * s;

            // ---- values of the chunk (independent of the prep group) ------------
            constexpr int kPerV = 64 * (D / 8) / kGroup;
            uint4 vv[kPerV];
#pragma unroll
            for (int it = 0; it < kPerV; ++it) {
                const int e = tid + it * kGroup;
                const int r = e / (D / 8), cc = e % (D / 8);
                const size_t row = static_cast<size_t>(tok0 + min(r, n - 1));  // always a row of this chunk
                vv[it] = __ldg(reinterpret_cast<const uint4 *>(a.v + row * ldv + static_cast<size_t>(h) * D + cc * 8));
            }

            // ---- wait for the chunk's operands ---------------------------------
            // (a failed wait is agreed on at the S1 barrier below)
            const bool ok_ready = __all_sync(0xffffffffu, mbar_wait_bounded(ready + s, (c >> 1) & 1));
            tc::fence_after_sync();

            // ---- S1: D1 = S0^T [Q;K]^T --------------------------------------------
            if (tid == 0 && ok_ready) {
                const uint64_t dQK = tc::desc_k_sw128(tc::smem_u32(sQK(qs)));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * 128 * 128 + (kk & 3) * 32) >> 4;
                    tc::mma_f16(d1, dS0T + off, dQK + off, kIdN128, kk > 0);
                }
                tc::mma_commit(mma_bar);
            }
            __syncwarp();
            if (tid < 64 && ok_ready) sGamC(s)[tid & 63] = sGam(s)[tid & 63];  // kept for the output of this chunk
            // values -> staging tile (the U^T tile is free until C4 of this chunk)
#pragma unroll
            for (int it = 0; it < kPerV; ++it) {
                const int e = tid + it * kGroup;
                const int r = e / (D / 8), cc = e % (D / 8);
                *reinterpret_cast<uint4 *>(sVst + r * D + cc * 8) = r < n ? vv[it] : make_uint4(0, 0, 0, 0);
            }

            // ---- output of the previous chunk while S1 runs ---------------------
            if (c > 0) output(s ^ 1, prev_n, prev_tok0);

            // ---- C2: V'^T = V^T - (K S0)^T diag(gamma) --------------------------
            const bool ok1 = mbar_wait_bounded(mma_bar, mma_phase);
            mma_phase ^= 1u;
            if (group_any(kBarChain, !ok1 || !ok_ready)) {
                failed = true;
                break;
            }
            tc::fence_after_sync();
            if (j < D) {
                float ks[32];
                tmem_load_row<32>(d1_lane + 64 + 32 * hf, ks);
                const float *gam = sGam(s) + 32 * hf;
#pragma unroll
                for (int i4 = 0; i4 < 32; i4 += 4) {
                    const float4 g4 = *reinterpret_cast<const float4 *>(gam + i4);
                    const float gg[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int i = i4 + u;
                        ks[i] = __uint_as_float(static_cast<uint32_t>(sVst[(32 * hf + i) * D + jm]) << 16) - gg[u] * ks[i];
                    }
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) store_chunk8_f16(sVpT, 128, jm, 4 * hf + q, ks + 8 * q);
            }
            tc::fence_proxy_async_smem();
            tc::fence_before_sync();
            group_sync(kBarChain);
            if (tid == 0) {
                tc::fence_after_sync();
                const uint64_t dT = tc::desc_k_sw128(tc::smem_u32(sTpp(s)));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) tc::mma_f16(d1 + 64, dVpT + kk * 2, dT + kk * 2, kIdN64, kk > 0);
                tc::mma_commit(mma_bar);
            }
            __syncwarp();
            if (j < D) {  // gamma_C scales the state while S3 runs
                const float gC = sGam(s)[63];
#pragma unroll 1
                for (int c0 = hf * kHalfD; c0 < (hf + 1) * kHalfD; c0 += 32) {
                    uint32_t r[32];
                    tc::tmem_ld32(my_lane + kColD5 + c0, r);
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(gC * __uint_as_float(r[i]));
                    tc::tmem_st32(my_lane + kColD5 + c0, r);
                }
            }
            tc::fence_before_sync();

            // ---- C4: U^T and (diag(dec) U)^T to fp16; D5 += (diag(dec) U)^T K, D6 = U^T P^T
            // (a failed wait is agreed on at the barrier that follows the phase;
            // the V'^T tile is free once S3 has completed)
            const bool ok2 = __all_sync(0xffffffffu, mbar_wait_bounded(mma_bar, mma_phase));
            mma_phase ^= 1u;
            tc::fence_after_sync();
            if (ok2 && j < D) {
                float u[32];
                tmem_load_row<32>(d1_lane + 64 + 32 * hf, u);
#pragma unroll
                for (int q = 0; q < 4; ++q) store_chunk8_f16(sUT, 128, jm, 4 * hf + q, u + 8 * q);
                const float *dec = sDec(s) + 32 * hf;
#pragma unroll
                for (int i4 = 0; i4 < 32; i4 += 4) {
                    const float4 d4 = *reinterpret_cast<const float4 *>(dec + i4);
                    u[i4] *= d4.x;
                    u[i4 + 1] *= d4.y;
                    u[i4 + 2] *= d4.z;
                    u[i4 + 3] *= d4.w;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) store_chunk8_f16(sVpT, 128, jm, 4 * hf + q, u + 8 * q);
            }
            tc::fence_proxy_async_smem();
            tc::fence_before_sync();
            if (group_any(kBarChain, !ok2)) {
                failed = true;
                break;
            }
            if (tid == 0) {
                tc::fence_after_sync();
                // K rows of the Q/K slot as B (N = key index i, K = token t), MN-major:
                // 64-column boxes 16 KB apart, a 16-token K step is 2048 B.
                const uint64_t dK = tc::desc_mn_sw128(tc::smem_u32(sQK(qs) + 8192), 16384);
                const uint64_t dPs = tc::desc_k_sw128(tc::smem_u32(sP(s)));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma_f16(tbase + kColD5, dVpT + kk * 2, dK + kk * (2048 >> 4), kIdNDbmn, 1);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) tc::mma_f16(tbase + kColD6, dUT + kk * 2, dPs + kk * 2, kIdN64, kk > 0);
                tc::mma_commit(mma_bar);
            }
            __syncwarp();

            // ---- C6: new state -> S0^T tile, emission, final state -----------------
            const bool ok3 = __all_sync(0xffffffffu, mbar_wait_bounded(mma_bar, mma_phase));
            mma_phase ^= 1u;
            tc::fence_after_sync();
            if (ok3) mbar_arrive(freeb + s);  // every MMA and read of this chunk's stage and Q/K slot is done
            if (ok3 && j < D) {
                float *ep = nullptr;
                if (E > 0 && n == kChunk && ((c + 1) % E) == 0) {
                    if (a.emit_table) {  // emission k of this sequence -> its cache block's slot
                        const int64_t col = static_cast<int64_t>(emit_first) + (c + 1) / E - 1;
                        const int slot = (col >= 0 && col < a.emit_table_stride)
                                             ? a.emit_table[static_cast<int64_t>(seq) * a.emit_table_stride + col]
                                             : static_cast<int>(a.num_slots);
                        if (slot >= 0 && slot < a.num_slots)
                            ep = a.state + ((static_cast<size_t>(slot) * a.h_v + h) * D + jm) * D;
                        else if (slot >= 0 && tid == 0)
                            report(a.dev_status, GDN_DEV_BAD_SLOT);
                    } else if (a.chunk_states) {
                        const int64_t idx = eoff + (c + 1) / E - 1;
                        if (idx >= 0 && idx < a.chunk_capacity)
                            ep = a.chunk_states + ((static_cast<size_t>(idx) * a.h_v + h) * D + jm) * D;
                    }
                }
                float *dp = (c == n_chunks - 1 && dst >= 0)
                                ? a.state + ((static_cast<size_t>(dst) * a.h_v + h) * D + jm) * D
                                : nullptr;
#pragma unroll 1
                for (int c0 = hf * kHalfD; c0 < (hf + 1) * kHalfD; c0 += 32) {
                    uint32_t r[32];
                    tc::tmem_ld32(my_lane + kColD5 + c0, r);
                    store_f16_chunks32(sS0T, jm, c0, r);
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        const float4 v = make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]),
                                                     __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
                        if (ep) __stcg(reinterpret_cast<float4 *>(ep + c0 + i), v);
                        if (dp) __stcg(reinterpret_cast<float4 *>(dp + c0 + i), v);
                    }
                }
            }
            tc::fence_proxy_async_smem();
            tc::fence_before_sync();
            if (group_any(kBarChain, !ok3)) {
                failed = true;
                break;
            }
            prev_n = n;
            prev_tok0 = tok0;
        }
        if (!failed && n_chunks > 0) output((n_chunks - 1) & 1, prev_n, prev_tok0);
        if (failed) {
            if (tid == 0) {
                report(a.dev_status, GDN_DEV_TIMEOUT);
                atomicExch(fail, 1);
            }
            // MMAs already issued get a bounded time to finish before the TMEM
            // they write is released.
            mbar_wait_bounded(mma_bar, mma_phase);
        }
    } else {
        // ============================= prep group ==============================
        // Thread (p, hf): TMEM lane / Gram row p, half hf of the row's work.
        const int pid = tid - kGroup;  // 0..255
        const int p = pid & 127, hf = pid >> 7;
        bool failed = false;
        const uint32_t aIdGram = tc::idesc_f16_f32acc(128, 64);
        // q, k of a chunk go straight into its Q/K slot by TMA (bf16, 128-byte
        // swizzle: the layout the MMA descriptors expect), issued at the start
        // of the previous chunk's preparation; g, beta into registers at the
        // same time.  The bf16 -> fp16 conversion runs in place, during the
        // previous chunk's diagonal solve, by the warps that solve nothing.
        constexpr uint32_t kTmaBytes = 2u * (D / 64) * 64 * 128;
        float gv = 0.f, bv = 0.f;
        auto load_gb = [&](int cc) {
            const int tk = t0 + cc * kChunk;
            const int nn = min(kChunk, Lseq - cc * kChunk);
            if (pid < 64) {
                const size_t gi = static_cast<size_t>(tk + min(pid & 63, nn - 1)) * a.h_v + h;
                gv = a.g[gi];
                bv = a.beta[gi];
            }
        };
        auto issue_tma = [&](int cc) {
            const int tk = t0 + cc * kChunk;
            if (pid == 0) {
                const int slot = cc % 3;
                uint8_t *tile = sQK(slot);
                uint64_t *tb = tma_bar + slot;
                mbar_expect_tx(tb, kTmaBytes);
#pragma unroll
                for (int kb = 0; kb < D / 64; ++kb) {
                    tma_load_2d(tile + kb * 16384, &L.tm_q, kh * D + kb * 64, tk, tb);
                    tma_load_2d(tile + kb * 16384 + 8192, &L.tm_k, kh * D + kb * 64, tk, tb);
                }
            }
        };
        // Waits for chunk cc's copies and converts its slot to fp16 in place
        // (16-byte items first_e, first_e + step, ...); rows past the sequence
        // end (the next sequence's tokens) become zeros.
        auto convert = [&](int cc, int first_e, int step) -> bool {
            const int slot = cc % 3;
            const int nn = min(kChunk, Lseq - cc * kChunk);
            uint8_t *tile = sQK(slot);
            if (!mbar_wait_bounded(tma_bar + slot, (cc / 3) & 1)) return false;
            for (int e = first_e; e < 64 * (D / 8); e += step) {
                const int r = e / (D / 8), c8 = e % (D / 8);
                uint4 *pq = reinterpret_cast<uint4 *>(tile + tc::sw128_chunk_offset(r, c8, 128));
                uint4 *pk = reinterpret_cast<uint4 *>(tile + tc::sw128_chunk_offset(64 + r, c8, 128));
                const uint4 z = make_uint4(0, 0, 0, 0);
                const uint4 xq = *pq, xk = *pk;
                *pq = r < nn ? bf16x8_to_f16x8(xq) : z;
                *pk = r < nn ? bf16x8_to_f16x8(xk) : z;
            }
            tc::fence_proxy_async_smem();  // the converted tile is read by the tensor cores
            return true;
        };
        if (n_chunks > 0) {
            issue_tma(0);
            if (n_chunks > 1) issue_tma(1);
            load_gb(0);
            if (!convert(0, pid, kGroup)) failed = true;
        }
        if (group_any(kBarPrep, failed)) failed = true;
        for (int c = 0; c < n_chunks && !failed; ++c) {
            const int s = c & 1, qs = c % 3;
            const int tok0 = t0 + c * kChunk;
            const int n = min(kChunk, Lseq - c * kChunk);
            // ---- next chunk's copies (each chunk's tile is converted one chunk ahead)
            uint8_t *qk = sQK(qs);
            bool okt;
            {
                if (pid < 64) {  // g, beta of this chunk, loaded one chunk ahead
                    const int t = pid & 63;
                    sGraw[t] = t < n ? gv : 0.f;
                    sBeta[t] = t < n ? bv : 0.f;
                }
                // The next chunk's Q/K slot and this chunk's stage were both last
                // used by chunk c - 2: one wait, by the issuing thread, covers
                // both (the group barrier below orders every write of the stage
                // after it).  Chunk 1's copies were issued with chunk 0's.
                bool okf = true;
                if (pid == 0 && c >= 2) okf = mbar_wait_bounded(freeb + s, ((c - 2) >> 1) & 1);
                if (c >= 1 && c + 1 < n_chunks && okf) issue_tma(c + 1);
                if (c + 1 < n_chunks) load_gb(c + 1);
                if (c + 2 < n_chunks && pid < 128) {  // q, k rows of chunk c + 2 into L2
                    const int rn = min(kChunk, Lseq - (c + 2) * kChunk);
                    const int r = pid & 63;
                    if (r < rn) {
                        const size_t row = static_cast<size_t>(tok0 + 2 * kChunk + r);
                        const uint16_t *src_row = (pid < 64 ? a.q : a.k) + row * ldq + kh * D;
                        asm volatile("prefetch.global.L2 [%0];" ::"l"(src_row) : "memory");
                        if (D > 64) asm volatile("prefetch.global.L2 [%0];" ::"l"(src_row + 64) : "memory");
                    }
                }
                okt = okf;
            }
            tc::fence_before_sync();
            if (group_any(kBarPrep, !okt)) {  // chunk c - 2 never finished: stop (bounded)
                failed = true;
                break;
            }
            // ---- Gram [Q;K] K^T (issued by warp 9 while warp 8 runs the prefix sum) --
            if (pid == 32) {
                tc::fence_after_sync();
                const uint64_t dQK = tc::desc_k_sw128(tc::smem_u32(qk));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * 128 * 128 + (kk & 3) * 32) >> 4;
                    tc::mma_f16(tbase + kColGram, dQK + off, dQK + off + (64 * 128 >> 4), aIdGram, kk > 0);
                }
                tc::mma_commit(gram_bar);
            }
            if (pid < 32) {  // inclusive prefix sum of g over the chunk, fixed order
                const int l = pid & 31;
                const float g0 = sGraw[2 * l], g1 = sGraw[2 * l + 1];
                const float pair = g0 + g1;
                float incl = pair;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (l >= o) incl += y;
                }
                const float excl = incl - pair;
                const float G0 = excl + g0, G1 = excl + g0 + g1;
                const float Gc = __shfl_sync(0xffffffffu, G1, 31);  // G_63, the chunk total
                sG[2 * l] = G0;
                sG[2 * l + 1] = G1;
                sGam(s)[2 * l] = expf(G0);
                sGam(s)[2 * l + 1] = expf(G1);
                sDec(s)[2 * l] = expf(Gc - G0);
                sDec(s)[2 * l + 1] = expf(Gc - G1);
            }
            group_sync(kBarPrep);  // g cumsum, gamma, dec visible
            __syncwarp();
            // Each warp reads the Gram only once every lane saw it complete; a
            // failure is agreed on at the barrier after P and A.
            const bool okg = __all_sync(0xffffffffu, mbar_wait_bounded(gram_bar, c & 1));
            tc::fence_after_sync();

            // ---- P rows (lanes 0..63) and A rows (lanes 64..127), columns 32 hf.. ----
            // Rows 0..31 x columns 32..63 are masked (warp-uniform): P gets zeros,
            // the upper triangle of A is never read.
            if (!okg) {
                // nothing: the barrier below ends the loop
            } else if (hf == 1 && (p & 32) == 0) {
                if (p < 64) {
                    const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int q = 4; q < 8; ++q)
                        *reinterpret_cast<uint4 *>(sP(s) + tc::sw128_chunk_offset(p & 63, q, 64)) = z;
                }
            } else {
                float x[32];
                tmem_load_row<32>(my_lane + kColGram + 32 * hf, x);
                const int r = p & 63;
                const float Gr = sG[r];
#pragma unroll
                for (int q4 = 0; q4 < 32; q4 += 4) {
                    const int q0 = 32 * hf + q4;
                    const float4 g4 = *reinterpret_cast<const float4 *>(sG + q0);
                    x[q4 + 0] = (q0 + 0 <= r) ? __expf(Gr - g4.x) * x[q4 + 0] : 0.f;
                    x[q4 + 1] = (q0 + 1 <= r) ? __expf(Gr - g4.y) * x[q4 + 1] : 0.f;
                    x[q4 + 2] = (q0 + 2 <= r) ? __expf(Gr - g4.z) * x[q4 + 2] : 0.f;
                    x[q4 + 3] = (q0 + 3 <= r) ? __expf(Gr - g4.w) * x[q4 + 3] : 0.f;
                }
                if (p < 64) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) store_chunk8_f16(sP(s), 64, r, 4 * hf + q, x + 8 * q);
                } else {
                    const float br = sBeta[r];
#pragma unroll
                    for (int q = 0; q < 32; q += 4) {
                        const int q0 = 32 * hf + q;
                        *reinterpret_cast<float4 *>(sM + r * kLdM + q0) =
                            make_float4(q0 + 0 < r ? br * x[q + 0] : 0.f, q0 + 1 < r ? br * x[q + 1] : 0.f,
                                        q0 + 2 < r ? br * x[q + 2] : 0.f, q0 + 3 < r ? br * x[q + 3] : 0.f);
                    }
                }
            }
            tc::fence_before_sync();
            if (group_any(kBarPrep, !okg)) {
                failed = true;
                mbar_wait_bounded(gram_bar, c & 1);  // let an issued Gram finish before TMEM is freed
                break;
            }

            // ---- T = (I + A)^-1: diagonal blocks, then level 1 || next chunk's Q/K to fp16
            // A diagonal block is solved and stored by the 16 lanes of one half
            // warp (warps 8 and 9): a warp barrier orders its reads before the
            // store, and the same warp then builds level 1 of the off-diagonal
            // part; the group barrier below orders both before level 2.
            bool okn = true;
            if (pid < 64) {
                float xd[16];
                invert_diag_solve(sM, pid, xd);
                __syncwarp();
                invert_diag_store(sM, pid, xd, sTpp(s), sBeta);
                __syncwarp();  // warp 8 holds blocks 0, 1 and warp 9 blocks 2, 3: level 1 per warp
                if (pid < 32) level1_warp<1>(sM, sW, pid & 31, sTpp(s), sBeta);
                else level1_warp<3>(sM, sW, pid & 31, sTpp(s), sBeta);
            } else if (c + 1 < n_chunks) {
                okn = convert(c + 1, pid - 64, kGroup - 64);
            }
            if (group_any(kBarPrep, !okn)) {  // diagonal blocks and level 1 visible to level 2
                failed = true;
                break;
            }
            // T'' = T diag(beta) is written as fp16 by the inverse itself.
            invert_offdiag(sM, sW, pid, sTpp(s), sBeta);
            tc::fence_proxy_async_smem();
            mbar_arrive(ready + s);
            group_sync(kBarPrep);  // scratch reuse by the next chunk
        }
        if (failed && pid == 0) {
            report(a.dev_status, GDN_DEV_TIMEOUT);
            atomicExch(fail, 1);
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tbase, kTmemCols);
}

template <int D>
cudaError_t launch_d(const PrefillLaunch &L, cudaStream_t stream) {
    const uint32_t smem = Smem<D>::kAlloc;
    cudaError_t e = cudaFuncSetAttribute(prefill_chunk_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    prefill_chunk_tc_kernel<D><<<L.a.num_seqs * L.a.h_v, kThreads, smem, stream>>>(L);
    return cudaGetLastError();
}

}  // namespace

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library); resolved once.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// rows x cols bf16, row-major with row stride cols; boxes of 64 rows x 64 cols.
bool encode_rows(CUtensorMap *m, const uint16_t *base, uint64_t rows, uint64_t cols) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {cols, rows > 0 ? rows : 1};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, 64};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_prefill(const PrefillArgs &a, int d, const int32_t *cu_host, cudaStream_t stream) {
    if (a.num_seqs == 0) return cudaSuccess;
    static_assert(sizeof(PrefillLaunch) < 32000, "kernel parameter size");
    // Longest sequences first, so the longest chains start in the first wave.
    PrefillLaunch L;
    L.a = a;
    const uint64_t cols = static_cast<uint64_t>(a.h_k) * d;
    if (a.total_tokens > 0 && (!encode_rows(&L.tm_q, a.q, a.total_tokens, cols) ||
                               !encode_rows(&L.tm_k, a.k, a.total_tokens, cols)))
        return cudaErrorNotSupported;
    L.n_order = a.num_seqs < kMaxOrder ? a.num_seqs : kMaxOrder;
    for (int i = 0; i < L.n_order; ++i) L.order[i] = i;
    for (int i = 1; i < L.n_order; ++i) {  // insertion sort by length, descending, stable
        const int v = L.order[i];
        const int lv = cu_host[v + 1] - cu_host[v];
        int k = i - 1;
        while (k >= 0 && (cu_host[L.order[k] + 1] - cu_host[L.order[k]]) < lv) {
            L.order[k + 1] = L.order[k];
            --k;
        }
        L.order[k + 1] = v;
    }
    return d == 128 ? launch_d<128>(L, stream) : launch_d<64>(L, stream);
}

}  // namespace gdn
