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
// For a chunk of C = 64 tokens entering with state S (d_k x d_v), local index
// t, G_t = sum_{s<=t} g_s, gamma_t = exp(G_t):
//
//     A_ts = beta_t exp(G_t - G_s) k_t.k_s  (s < t),   T = (I + A)^-1
//     T''  = T diag(beta),   T''' = T diag(beta gamma),   W = T''' K
//     U    = T'' V - W S                                      (rows u_t)
//     O    = Q~ S + P~ U,   Q~_t = scale gamma_t q_t,  P~_ts = scale exp(G_t - G_s) q_t.k_s (s <= t)
//     S'   = gamma_C S + K^T diag(dec) U,   dec_t = exp(G_C - G_t)
//
// Only the products with S depend on the carried state; everything else
// (Gram, decays, P~, A, the inverse, T'', W, the fp16 operand tiles) is local
// to the chunk.  One CTA runs one (sequence, value head) chain, in two warp
// groups:
//
//   chain group (warps 0-7; thread (j, hf): TMEM lane j = value column j,
//     half hf of the lane's columns), per chunk:
//       D_U  += S16^T (-W)^T          (D_U was preset to U'^T = V^T T''^T)
//       D_O   = S16^T Q~^T            (output accumulator)
//       U^T, (diag(dec) U)^T -> fp16 A operands in TMEM
//       D_S   = gamma_C D_S + (diag(dec) U)^T K,   D_O += U^T P~^T
//       D_S  -> fp16 S16 (A operand in TMEM), emission, final state
//     writes the previous chunk's output while the first products run (the
//     output product of the chunk waits for it), converts the next chunk's
//     q~, k, v tiles to fp16 in place (after their Gram has read them) while
//     the state update runs, and then queues the Gram [Q;K] K^T of the chunk
//     after next (bf16, straight from its TMA tile, into its own TMEM columns);
//   prep group (warps 8-15), one chunk ahead: q, k, v tiles by TMA (and the
//     first chunk's Gram), decays, P~ and A from the Gram, the
//     inverse (16x16 diagonal blocks by substitution and the first doubling
//     level on the CUDA cores in fp32; the second level, the 32x32 lower-left
//     block, as two tcgen05 products), T'' and -T''' (U'^T = V^T T''^T is
//     then preset by the chain's tensor-core issuer), and
//     -W^T = K^T (-T''')^T.
//
// The fp32 state lives in TMEM for the whole chain; its fp16 copy (an operand)
// is written once per chunk.  A chunk's arithmetic depends only on its own
// inputs and the fp32 state entering it, so results do not depend on the
// batch, and restarting from an emitted state reproduces the uninterrupted
// run bit for bit.
//
// Every wait is bounded.  A wait that runs out sets GDN_DEV_TIMEOUT, both
// groups agree on the failure at their next group barrier and leave their
// loops, and before TMEM is released the threads that issued asynchronous
// work wait (again bounded) for every MMA and TMA copy still in flight.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

#ifndef GDN_WAIT_CYCLES
#define GDN_WAIT_CYCLES 2000000000LL
#endif

namespace gdn {
namespace {

constexpr int kThreads = 512;  // chain group + prep group
constexpr int kGroup = 256;
constexpr int kBarChain = 1;  // named barrier ids (0 is __syncthreads)
constexpr int kBarPrep = 2;
constexpr int kBarPairL1 = 3;  // 3, 4: warps 8 + 12, 9 + 13 (first inverse level)
// Limit of every handshake wait between the groups, in SM clock cycles
// (~1 s by default); a build may shorten it to exercise the failure path.
constexpr long long kWaitCycles = GDN_WAIT_CYCLES;
// Limit of the waits for work already in flight when a chain stops (~1 s).
constexpr long long kDrainCycles = 2000000000LL;
constexpr int kMaxOrder = 2048;

struct PrefillLaunch {
    CUtensorMap tm_q, tm_k;  // q, k as 2-D [T][h_k d] bf16, 64 x 64 boxes, 128-byte swizzle
    CUtensorMap tm_v;        // v as 2-D [T][h_v d] bf16, same boxes
    PrefillArgs a;
    int32_t n_order;
    int32_t order[kMaxOrder];  // launch rank -> sequence, longest first
};

// Row stride of the 64x64 fp32 inverse scratch: 68 floats keep 16-byte
// alignment and put 8 consecutive rows on disjoint bank quads.
constexpr int kLdM = 68;

template <int D>
struct Smem {
    // Operand tiles (128-byte swizzle, 1024-aligned).
    static constexpr uint32_t kQKBytes = 256u * D;  // per 64-wide block of d: q box (8 KB), k box (8 KB)
    static constexpr uint32_t kQK0 = 0;             // ring of three slots
    static constexpr uint32_t kVBytes = 128u * D;   // v boxes, 8 KB apart
    static constexpr uint32_t kV0 = kQK0 + 3 * kQKBytes;  // ring of two slots
    static constexpr uint32_t kWT = kV0 + 2 * kVBytes;    // -W^T [i][t] fp16 (MN-major B of S16 (-W)^T)
    static constexpr uint32_t kP0 = kWT + 128u * D;       // P~ [t][s] fp16, two stages
    static constexpr uint32_t kTpp = kP0 + 16384;         // T'' [t][s] fp16
    static constexpr uint32_t kTppp = kTpp + 8192;        // -T''' [t][s] fp16
    static constexpr uint32_t kL2A1 = kTppp + 8192;       // A_B (rows 32..63, cols 0..31 of A), K-major
    static constexpr uint32_t kL2B1 = kL2A1 + 4096;       // T_top, MN-major B
    static constexpr uint32_t kL2A2 = kL2B1 + 4096;       // T_bot, K-major
    static constexpr uint32_t kL2B2 = kL2A2 + 4096;       // -X = -(A_B T_top), MN-major B
    // Plain buffers.
    static constexpr uint32_t kM = kL2B2 + 4096;          // f32 [64][kLdM]: A, then T
    static constexpr uint32_t kWb = kM + 64 * kLdM * 4;   // f32 [2][16][16] level-1 products
    static constexpr uint32_t kGl = kWb + 4096;           // f32 [64] cumulative log decay G, times log2(e)
    static constexpr uint32_t kGam = kGl + 256;           // f32 [64] gamma
    static constexpr uint32_t kBG = kGam + 256;           // f32 [64] beta gamma
    static constexpr uint32_t kBeta = kBG + 256;          // f32 [64]
    static constexpr uint32_t kDec = kBeta + 256;         // f32 [2][64] exp(G_C - G_t), per stage
    static constexpr uint32_t kGc = kDec + 512;           // f32 [2] gamma_C, per stage
    static constexpr uint32_t kBars = kGc + 16;           // 21 mbarriers
    static constexpr uint32_t kTmem = kBars + 21 * 8;     // TMEM base address
    static constexpr uint32_t kFail = kTmem + 4;          // int
    static constexpr uint32_t kEoff = kFail + 12;         // long long [16]
    static constexpr uint32_t kBytes = kEoff + 128;
    static constexpr uint32_t kAlloc = kBytes + 1024;     // + alignment slack
    static_assert(kV0 % 1024 == 0 && kWT % 1024 == 0 && kP0 % 1024 == 0 && kTpp % 1024 == 0, "");
    static_assert(kL2A1 % 1024 == 0 && kL2A2 % 1024 == 0 && kL2B1 % 1024 == 0 && kL2B2 % 1024 == 0, "");
    // A level-2 MMA reads 128 rows (16 KB) of its A tile; rows past 31 are
    // don't-care but must lie inside the allocation.
    static_assert(kL2A2 + 16384 <= kBytes, "");
    static_assert(kM % 16 == 0 && kWb % 16 == 0 && kBars % 8 == 0 && kEoff % 8 == 0, "");
    static_assert(kAlloc <= 232448, "shared memory budget");
};

// TMEM column map (512 columns; lane j = value column j, or row of a prep product).
constexpr uint32_t kColS = 0;       // fp32 state S^T, D columns
constexpr uint32_t kColU = 128;     // U^T, 64 columns
constexpr uint32_t kColO = 192;     // output accumulator O^T, 64 columns
constexpr uint32_t kColGram = 256;  // Gram [Q;K] K^T of a chunk, 64 columns
constexpr uint32_t kColS16 = 320;   // S^T fp16, packed (D / 2 columns): A operand
constexpr uint32_t kColU16 = 384;   // U^T fp16 packed: A operand
constexpr uint32_t kColUd16 = 416;  // (diag(dec) U)^T fp16 packed: A operand
constexpr uint32_t kColPrep = 448;  // prep products: X and T_B; -W^T
constexpr uint32_t kTmemCols = 512;

// mbarriers.
enum : int {
    kBarTmaQK = 0,   // [3] q/k slot loaded
    kBarTmaV = 3,    // [2] v slot loaded
    kBarGram = 5,    // Gram done
    kBarL2 = 6,      // level-2 products done (two per chunk)
    kBarW = 7,       // -W^T done
    kBarUReady = 8,  // T'' and v of the next chunk ready (chain may preset U'^T)
    kBarReady = 9,   // [2] a chunk's operands ready for the chain
    kBarA = 11,      // chain: D_U complete
    kBarC = 12,      // chain: state update and output complete
    kBarWFree = 13,  // chain done reading -W^T
    kBarTFree = 14,  // chain done reading T'' and its v slot
    kBarQKFree = 15, // chain done reading a q/k slot and its P~ / decay stage
    kBarDrainC = 16,
    kBarDrainP = 17,
    kBarGamReady = 18, // decays of the chunk the prep group works on are in shared memory
    kBarConvDone = 19, // chain group: q~, k, v of that chunk converted to fp16
    kBarGramFree = 20, // prep group done reading a chunk's Gram from TMEM
    kNumBars = 21
};

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// 8 bf16 (one uint4) -> 8 fp16 times f (exact for f = 1 except below 2^-14).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 w, float f) {
    uint4 r;
    r.x = pack_half2(f * __uint_as_float(w.x << 16), f * __uint_as_float(w.x & 0xffff0000u));
    r.y = pack_half2(f * __uint_as_float(w.y << 16), f * __uint_as_float(w.y & 0xffff0000u));
    r.z = pack_half2(f * __uint_as_float(w.z << 16), f * __uint_as_float(w.z & 0xffff0000u));
    r.w = pack_half2(f * __uint_as_float(w.w << 16), f * __uint_as_float(w.w & 0xffff0000u));
    return r;
}

// 8 bf16 (one uint4) -> 8 fp16 (exact except below 2^-14).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 w) {
    uint4 r;
    r.x = pack_half2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u));
    r.y = pack_half2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
    r.z = pack_half2(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xffff0000u));
    r.w = pack_half2(__uint_as_float(w.w << 16), __uint_as_float(w.w & 0xffff0000u));
    return r;
}

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
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}

// (a, b) * (s, t) as one packed fp32x2 multiply (round to nearest, as two
// separate fp32 multiplies would give).
__device__ __forceinline__ void mul2(uint32_t &a, uint32_t &b, float s, float t) {
    asm("{\n\t.reg .b64 x, f, y;\n\t"
        "mov.b64 x, {%0, %1};\n\t"
        "mov.b64 f, {%2, %3};\n\t"
        "mul.rn.f32x2 y, x, f;\n\t"
        "mov.b64 {%0, %1}, y;\n\t}"
        : "+r"(a), "+r"(b)
        : "f"(s), "f"(t));
}

// 2^x by the hardware approximation (the operation __expf is built on).
__device__ __forceinline__ float exp2f_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Byte offset of 16-byte chunk c (8 fp16 along N) of row k of an MN-major
// SW128 tile (rows are the K index, 64 N elements per 128-byte row).
__device__ __forceinline__ uint32_t mn_chunk_offset(uint32_t k, uint32_t c) {
    return (k >> 3) * 1024u + (k & 7u) * 128u + (((c & 7u) ^ (k & 7u)) << 4);
}

// Bounded wait for the phase of `bar` with the given parity; gives up as
// soon as any thread has flagged a failure, and flags one when it runs out.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, int *fail) {
    const long long start = clock64();
    while (!tc::mbar_try_wait(bar, parity)) {
        if (*reinterpret_cast<volatile int *>(fail)) return false;
        if (clock64() - start > kWaitCycles) {
            atomicExch(fail, 1);
            return false;
        }
    }
    return true;
}
// Bounded wait for work already in flight (ignores the failure flag).
__device__ __forceinline__ bool drain_bar(uint64_t *bar, uint32_t parity) {
    const long long start = clock64();
    while (!tc::mbar_try_wait(bar, parity))
        if (clock64() - start > kDrainCycles) return false;
    return true;
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

// Sum over s' < s of floor(L_s' / (64 E)), by the whole block.
__device__ int64_t emit_offset(const int32_t *cu, int s, int E, long long *part) {
    long long acc = 0;
    const long long per = static_cast<long long>(kChunk) * E;
    for (int i = threadIdx.x; i < s; i += blockDim.x) acc += (cu[i + 1] - cu[i]) / per;
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

// ---- the inverse, CUDA-core part ----------------------------------------------
// Diagonal 16x16 blocks of T = (I + A)^-1 for a strictly lower-triangular A
// held in M (fp32, row stride kLdM), by the 64 threads p < 64 (block
// p / 16, column c = p % 16), left-looking: x_i = [i == c] - sum_{j<i} A_ij x_j,
// which gives x_i = 0 above the diagonal since x_j = 0 for j < c.  Rows are
// read as float4 (shared-memory bandwidth is shared with the tensor cores'
// operand reads).  The column is written over the block's A entries after a
// warp barrier.
__device__ __forceinline__ void invert_diag_solve(const float *M, int p, float (&x)[16]) {
    const int c = p & 15, base = ((p >> 4) & 3) * 16;
    const float *row = M + base * kLdM + base;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
        for (int j4 = 0; j4 < i; j4 += 4) {
            const float4 m = *reinterpret_cast<const float4 *>(row + i * kLdM + j4);
            acc0 = fmaf(m.x, x[j4], acc0);
            if (j4 + 1 < i) acc1 = fmaf(m.y, x[j4 + 1], acc1);
            if (j4 + 2 < i) acc0 = fmaf(m.z, x[j4 + 2], acc0);
            if (j4 + 3 < i) acc1 = fmaf(m.w, x[j4 + 3], acc1);
        }
        x[i] = i == c ? 1.f : (i < c ? 0.f : -(acc0 + acc1));
    }
}
__device__ __forceinline__ void invert_diag_store(float *M, int p, const float (&x)[16]) {
    const int c = p & 15, base = ((p >> 4) & 3) * 16;
#pragma unroll
    for (int i = 0; i < 16; ++i) M[(base + i) * kLdM + base + c] = x[i];
}

__device__ __forceinline__ void fma4(float4 &acc, float a, const float4 &t) {
    acc.x = fmaf(a, t.x, acc.x);
    acc.y = fmaf(a, t.y, acc.y);
    acc.z = fmaf(a, t.z, acc.z);
    acc.w = fmaf(a, t.w, acc.w);
}
// acc += X[i][0..16) * Y[0..16)[4cq .. 4cq + 4) for 16x16 blocks X, Y.
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
// First doubling level: T_{B,B-1} = -T_BB (A_{B,B-1} T_{B-1,B-1}) in fp32,
// lane = (row i = lane / 2, column group cq of four columns).
// Half of it (columns 4 cq .. 4 cq + 3, cq = 2 (lane % 2) + u) by one warp,
// the other half (the other u) by a second warp, with barrier `bar` (64
// threads) around each step: before the first, the diagonal blocks are
// stored; between the two, both warps have read all of A_{B,B-1}, which the
// second step overwrites with T_{B,B-1}; after the second, all of T_{B,B-1}
// is in place.  Each warp reads back only its own part of Y.
__device__ __forceinline__ void pair_sync(int id) {  // two warps
    asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
}

template <int B>
__device__ __forceinline__ void level1_half(float *M, float *Wb, int lane, int u, int bar) {
    const int i = (lane >> 1) & 15, cq = 2 * (lane & 1) + u;
    float *Y = Wb + (B == 3 ? 256 : 0);
    pair_sync(bar);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    block_mac<kLdM, kLdM>(acc, M + (B * 16) * kLdM + (B - 1) * 16, M + ((B - 1) * 16) * kLdM + (B - 1) * 16, i, cq);
    *reinterpret_cast<float4 *>(Y + i * 16 + 4 * cq) = acc;
    pair_sync(bar);
    acc = make_float4(0.f, 0.f, 0.f, 0.f);
    block_mac<kLdM, 16>(acc, M + (B * 16) * kLdM + B * 16, Y, i, cq);
    *reinterpret_cast<float4 *>(M + (B * 16 + i) * kLdM + (B - 1) * 16 + 4 * cq) =
        make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
    pair_sync(bar);
}

// Writes 16 fp32 values v (columns 16q .. 16q + 15 of row t) as T'' = v beta
// and -T''' = -v beta gamma into the two 64-row K-major fp16 tiles.
__device__ __forceinline__ void store_t_segment(uint8_t *Tpp, uint8_t *Tppp, int t, int q, const float (&v)[16],
                                                const float *beta, const float *bg) {
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
        const int s0 = 16 * q + 8 * h2;
        uint4 a, b;
        a.x = pack_half2(v[8 * h2 + 0] * beta[s0 + 0], v[8 * h2 + 1] * beta[s0 + 1]);
        a.y = pack_half2(v[8 * h2 + 2] * beta[s0 + 2], v[8 * h2 + 3] * beta[s0 + 3]);
        a.z = pack_half2(v[8 * h2 + 4] * beta[s0 + 4], v[8 * h2 + 5] * beta[s0 + 5]);
        a.w = pack_half2(v[8 * h2 + 6] * beta[s0 + 6], v[8 * h2 + 7] * beta[s0 + 7]);
        b.x = pack_half2(-v[8 * h2 + 0] * bg[s0 + 0], -v[8 * h2 + 1] * bg[s0 + 1]);
        b.y = pack_half2(-v[8 * h2 + 2] * bg[s0 + 2], -v[8 * h2 + 3] * bg[s0 + 3]);
        b.z = pack_half2(-v[8 * h2 + 4] * bg[s0 + 4], -v[8 * h2 + 5] * bg[s0 + 5]);
        b.w = pack_half2(-v[8 * h2 + 6] * bg[s0 + 6], -v[8 * h2 + 7] * bg[s0 + 7]);
        const uint32_t off = tc::sw128_chunk_offset(t, 2 * q + h2, 64);
        *reinterpret_cast<uint4 *>(Tpp + off) = a;
        *reinterpret_cast<uint4 *>(Tppp + off) = b;
    }
}

// Writes 32 values (fp32 bit patterns, scaled by f) as the four 16-byte fp16
// chunks of a 32-column row: K-major row (`kmajor`) or MN-major row k.
__device__ __forceinline__ void store_row32_f16(uint8_t *tile, int row, const uint32_t (&x)[32], float f,
                                                bool kmajor) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 v;
        v.x = pack_half2(f * __uint_as_float(x[8 * q + 0]), f * __uint_as_float(x[8 * q + 1]));
        v.y = pack_half2(f * __uint_as_float(x[8 * q + 2]), f * __uint_as_float(x[8 * q + 3]));
        v.z = pack_half2(f * __uint_as_float(x[8 * q + 4]), f * __uint_as_float(x[8 * q + 5]));
        v.w = pack_half2(f * __uint_as_float(x[8 * q + 6]), f * __uint_as_float(x[8 * q + 7]));
        const uint32_t off = kmajor ? tc::sw128_chunk_offset(row, q, 128) : mn_chunk_offset(row, q);
        *reinterpret_cast<uint4 *>(tile + off) = v;
    }
}

// Gram [Q;K] K^T of one chunk in bf16, straight from its q/k TMA tile (q box,
// then k box, per 64-wide block of d), into the Gram TMEM columns; completion
// is signalled on `bar`.
template <int D>
__device__ __forceinline__ void gram_mma(uint32_t tbase, const uint8_t *qk_tile, uint64_t *bar) {
    const uint64_t dQK = tc::desc_k_sw128(tc::smem_u32(qk_tile));
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
        tc::mma_f16(tbase + kColGram, dQK + off, dQK + off + (8192 >> 4),
                    tc::idesc_f16_f32acc(128, 64) | tc::kIdescBf16, kk > 0);
    }
    tc::mma_commit(bar);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_chain_kernel(const __grid_constant__ PrefillLaunch L) {
    using SM = Smem<D>;
    constexpr int kKB = D / 64;                              // 64-wide blocks of d
    constexpr uint32_t kLboK = D == 128 ? 16384u : 0u;       // k box stride inside a q/k slot
    constexpr uint32_t kLboV = D == 128 ? 8192u : 0u;        // v box stride inside a v slot
    const PrefillArgs &a = L.a;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    auto sQK = [&](int slot) { return sm + SM::kQK0 + slot * SM::kQKBytes; };
    auto sV = [&](int slot) { return sm + SM::kV0 + slot * SM::kVBytes; };
    auto sP = [&](int st) { return sm + SM::kP0 + st * 8192; };
    auto sDec = [&](int st) { return reinterpret_cast<float *>(sm + SM::kDec + st * 256); };
    uint8_t *sWT = sm + SM::kWT, *sTpp = sm + SM::kTpp, *sTppp = sm + SM::kTppp;
    uint8_t *sL2A1 = sm + SM::kL2A1, *sL2B1 = sm + SM::kL2B1, *sL2A2 = sm + SM::kL2A2, *sL2B2 = sm + SM::kL2B2;
    float *sM = reinterpret_cast<float *>(sm + SM::kM), *sWb = reinterpret_cast<float *>(sm + SM::kWb);
    float *sGl = reinterpret_cast<float *>(sm + SM::kGl), *sGam = reinterpret_cast<float *>(sm + SM::kGam);
    float *sBG = reinterpret_cast<float *>(sm + SM::kBG), *sBeta = reinterpret_cast<float *>(sm + SM::kBeta);
    float *sGc = reinterpret_cast<float *>(sm + SM::kGc);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + SM::kBars);
    uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(sm + SM::kTmem);
    int *fail = reinterpret_cast<int *>(sm + SM::kFail);
    const volatile int *vfail = fail;
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
    const size_t ldv = static_cast<size_t>(a.h_v) * D;
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
        for (int b = 0; b < kNumBars; ++b) tc::mbar_init(bars + b, 1);
        *fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = *tmem_ptr;
    const uint32_t tl = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);  // this warp's TMEM lanes

    if (warp < 8) {
        // ============================ chain group ==============================
        const int j = tid & 127, hf = tid >> 7;
        const bool jv = j < D;  // warp-uniform: d = 64 leaves lane quarters 2, 3 without a column
        constexpr int kHalf = D / 2;
        const uint32_t idU = tc::idesc_f16_f32acc(128, 64);
        const uint32_t idS = tc::idesc_f16_f32acc(128, D) | tc::kIdescBmn;
        const uint64_t dWT = tc::desc_mn_sw128(tc::smem_u32(sWT), 0);
        bool failed = false;
        int prev_n = 0, prev_tok0 = 0;

        // Initial state row j (half hf): fp32 into D_S, fp16 into S16; for an
        // empty sequence straight to the destination slot.
        if (jv) {
            const float *sp = src >= 0 ? a.state + ((static_cast<size_t>(src) * a.h_v + h) * D + j) * D : nullptr;
            float *dp = (Lseq == 0 && dst >= 0) ? a.state + ((static_cast<size_t>(dst) * a.h_v + h) * D + j) * D
                                                : nullptr;
#pragma unroll 1
            for (int c0 = hf * kHalf; c0 < (hf + 1) * kHalf; c0 += 32) {
                uint32_t r[32], p16[16];
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
#pragma unroll
                for (int i = 0; i < 16; ++i) p16[i] = pack_half2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                if (Lseq > 0) {
                    tc::tmem_st32(tl + kColS + c0, r);
                    tc::tmem_st16(tl + kColS16 + c0 / 2, p16);
                }
            }
        } else if (hf == 0 && Lseq > 0) {  // d = 64: rows 64..127 of the A operands stay zero
            uint32_t z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0u;
            tc::tmem_st32(tl + kColS16, z);
            tc::tmem_st32(tl + kColU16, z);
            tc::tmem_st32(tl + kColUd16, z);
        }
        tc::fence_before_sync();
        group_sync(kBarChain);

        // U'^T = V^T T''^T into D_U for chunk cc (v slot cc & 1 as MN-major A).
        auto issue_u = [&](int cc) {
            const uint64_t dV = tc::desc_mn_sw128(tc::smem_u32(sV(cc & 1)), kLboV);
            const uint64_t dT = tc::desc_k_sw128(tc::smem_u32(sTpp));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                tc::mma_f16(tbase + kColU, dV + kk * (2048 >> 4), dT + kk * 2, idU | tc::kIdescAmn, kk > 0);
            tc::mma_commit(bars + kBarTFree);
        };

        // Output of a finished chunk, o_t = (Q~ S + P~ U)_t, tokens 32 hf ..
        // 32 hf + 31 of value column j, one bf16 per (token, j): a warp's 32
        // lanes store 64 contiguous bytes per token.
        auto output = [&](int n_out, int tok_out, int hh) {
            uint32_t r[32];
            tc::tmem_ld32(tl + kColO + 32 * hh, r);
            uint16_t *op = a.o + static_cast<size_t>(tok_out + 32 * hh) * ldv + static_cast<size_t>(h) * D + j;
            const int lim = n_out - 32 * hh;
#pragma unroll
            for (int i = 0; i < 32; ++i, op += ldv)
                if (i < lim) *op = float_to_bf16_bits(__uint_as_float(r[i]));
        };

        // ---- C0: q~, k, v of chunk cc to fp16 in place: after the Gram has read
        // the bf16 q/k tile.  Chunk 0 before the loop, chunk c + 1 while the
        // state update of chunk c runs on the tensor cores.  Thread tid owns the
        // 16-byte items tid and tid + 256 of every 64 x 64 box (rows tid / 8 and
        // tid / 8 + 32); rows past the sequence end become zeros; q is scaled by
        // scale gamma_t.  Returns false when the group fails.
        auto convert = [&](int cc) -> bool {
            const int ncc = min(kChunk, Lseq - cc * kChunk);
            uint8_t *qkc = sQK(cc % 3);
            bool ok0 = wait_bar(bars + kBarGram, cc & 1, fail) && wait_bar(bars + kBarGamReady, cc & 1, fail) &&
                       wait_bar(bars + kBarTmaQK + cc % 3, (cc / 3) & 1, fail) &&
                       wait_bar(bars + kBarTmaV + (cc & 1), (cc / 2) & 1, fail);
            if (ok0) {
                uint8_t *vt = sV(cc & 1);
                const int r0 = tid >> 3;
                const float f0 = a.scale * sGam[r0], f1 = a.scale * sGam[r0 + 32];
#pragma unroll
                for (int b = 0; b < 3 * kKB; ++b) {
                    const int kind = b / kKB, kb = b % kKB;
                    uint8_t *base = (kind == 2 ? vt + kb * 8192 : qkc + kb * 16384 + (kind == 1 ? 8192 : 0)) + tid * 16;
                    const uint4 x0 = *reinterpret_cast<const uint4 *>(base);
                    const uint4 x1 = *reinterpret_cast<const uint4 *>(base + 4096);
                    uint4 y0 = make_uint4(0, 0, 0, 0), y1 = make_uint4(0, 0, 0, 0);
                    if (r0 < ncc) y0 = kind == 0 ? bf16x8_to_f16x8(x0, f0) : bf16x8_to_f16x8(x0);
                    if (r0 + 32 < ncc) y1 = kind == 0 ? bf16x8_to_f16x8(x1, f1) : bf16x8_to_f16x8(x1);
                    *reinterpret_cast<uint4 *>(base) = y0;
                    *reinterpret_cast<uint4 *>(base + 4096) = y1;
                }
            }
            tc::fence_proxy_async_smem();  // read by the tensor cores
            if (group_any(kBarChain, !ok0 || *vfail)) return false;
            if (tid == 0) mbar_arrive(bars + kBarConvDone);
            return true;
        };

        // The Gram of chunk cc, queued by thread 0 once the conversion of chunk
        // cc - 1 is done and the prep group has read the Gram of chunk cc - 1
        // (so that neither still waits on the previous completion of kBarGram):
        // it runs behind the products already queued and is complete long
        // before the prep group needs it.
        auto issue_gram_ahead = [&](int cc) -> bool {
            if (!wait_bar(bars + kBarGramFree, (cc - 1) & 1, fail) ||
                !wait_bar(bars + kBarTmaQK + cc % 3, (cc / 3) & 1, fail))
                return false;
            tc::fence_after_sync();
            gram_mma<D>(tbase, sQK(cc % 3), bars + kBarGram);
            return true;
        };

        if (n_chunks > 0 && !convert(0)) failed = true;
        if (!failed && tid == 0 && n_chunks > 1 && !issue_gram_ahead(1)) atomicExch(fail, 1);
        for (int c = 0; c < n_chunks && !failed; ++c) {
            const int s = c & 1;
            const int tok0 = t0 + c * kChunk;
            const int n = min(kChunk, Lseq - c * kChunk);
            uint8_t *qk = sQK(c % 3);

            // ---- P0: operands of chunk c; D_U += S16^T (-W)^T, D_O = S16^T Q~^T --
            // (wait results that gate warp-collective TMEM accesses are made warp-uniform)
            const bool okr = __all_sync(0xffffffffu, wait_bar(bars + kBarReady + s, (c >> 1) & 1, fail));
            tc::fence_after_sync();
            if (tid == 0 && okr) {
                const bool oku = wait_bar(bars + kBarUReady, c & 1, fail);  // T'' (v of chunk c is converted already)
                if (oku) {
                    issue_u(c);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        tc::mma_f16_ta(tbase + kColU, tbase + kColS16 + kk * 8, dWT + kk * (2048 >> 4),
                                       idU | tc::kIdescBmn, 1);
                    tc::mma_commit(bars + kBarA);
                    tc::mma_commit(bars + kBarWFree);
                } else {
                    atomicExch(fail, 1);
                }
            }
            __syncwarp();
            // Warp 0 issues the products; warp 4 (same TMEM lanes) does both halves of
            // their lanes' output and state scaling.
            const int h_lo = warp == 4 ? 0 : hf, h_hi = warp == 4 ? 2 : hf + 1;
            if (c > 0 && jv && warp != 0)
                for (int hh = h_lo; hh < h_hi; ++hh) output(prev_n, prev_tok0, hh);
            if (jv && okr && warp != 0) {  // gamma_C scales the fp32 state while the products run
                const float gC = sGc[s];
#pragma unroll 1
                for (int c0 = h_lo * kHalf; c0 < h_hi * kHalf; c0 += 32) {
                    uint32_t r[32];
                    tc::tmem_ld32(tl + kColS + c0, r);
#pragma unroll
                    for (int i = 0; i < 32; i += 2) mul2(r[i], r[i + 1], gC, gC);
                    tc::tmem_st32(tl + kColS + c0, r);
                }
            }
            // The previous chunk's output has been read: D_O = S16^T Q~^T may start.
            tc::fence_before_sync();
            if (group_any(kBarChain, !okr || *vfail)) {
                failed = true;
                break;
            }
            if (tid == 0) {
                tc::fence_after_sync();
                const uint64_t dQ = tc::desc_k_sw128(tc::smem_u32(qk));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    tc::mma_f16_ta(tbase + kColO, tbase + kColS16 + kk * 8,
                                   dQ + (((kk >> 2) * 16384 + (kk & 3) * 32) >> 4), idU, kk > 0);
            }
            __syncwarp();
            const bool oka = __all_sync(0xffffffffu, okr && wait_bar(bars + kBarA, c & 1, fail));
            tc::fence_after_sync();

            // ---- P1: U^T and (diag(dec) U)^T to fp16 A operands --------------------
            if (oka && jv) {
                uint32_t r[32], pu[16], pd[16];
                tc::tmem_ld32(tl + kColU + 32 * hf, r);
                const float *dec = sDec(s) + 32 * hf;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    uint32_t u0 = r[2 * i], u1 = r[2 * i + 1];
                    pu[i] = pack_half2(__uint_as_float(u0), __uint_as_float(u1));
                    const float2 d2 = *reinterpret_cast<const float2 *>(dec + 2 * i);
                    mul2(u0, u1, d2.x, d2.y);
                    pd[i] = pack_half2(__uint_as_float(u0), __uint_as_float(u1));
                }
                tc::tmem_st16(tl + kColU16 + 16 * hf, pu);
                tc::tmem_st16(tl + kColUd16 + 16 * hf, pd);
            }
            tc::fence_before_sync();
            if (group_any(kBarChain, !oka || *vfail)) {
                failed = true;
                break;
            }

            // ---- P2: D_S += (diag(dec) U)^T K, D_O += U^T P~^T; preset next U'^T --
            if (tid == 0) {
                tc::fence_after_sync();
                const uint64_t dK = tc::desc_mn_sw128(tc::smem_u32(qk + 8192), kLboK);
                const uint64_t dPs = tc::desc_k_sw128(tc::smem_u32(sP(s)));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma_f16_ta(tbase + kColS, tbase + kColUd16 + kk * 8, dK + kk * (2048 >> 4), idS, 1);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma_f16_ta(tbase + kColO, tbase + kColU16 + kk * 8, dPs + kk * 2, idU, 1);
                tc::mma_commit(bars + kBarC);
                tc::mma_commit(bars + kBarQKFree);
            }
            __syncwarp();
            if (c + 1 < n_chunks && !convert(c + 1)) {  // the next chunk's operands, while these products run
                failed = true;
                break;
            }
            if (tid == 0 && c + 2 < n_chunks && !issue_gram_ahead(c + 2)) atomicExch(fail, 1);
            const bool okc = __all_sync(0xffffffffu, wait_bar(bars + kBarC, c & 1, fail));
            tc::fence_after_sync();

            // ---- P3: new state -> S16, emission, final state -------------------------
            if (okc && jv) {
                float *ep = nullptr;
                if (E > 0 && n == kChunk && ((c + 1) % E) == 0) {
                    if (a.emit_table) {  // emission k of this sequence -> its cache block's slot
                        const int64_t col = static_cast<int64_t>(emit_first) + (c + 1) / E - 1;
                        const int slot = (col >= 0 && col < a.emit_table_stride)
                                             ? a.emit_table[static_cast<int64_t>(seq) * a.emit_table_stride + col]
                                             : static_cast<int>(a.num_slots);
                        if (slot >= 0 && slot < a.num_slots)
                            ep = a.state + ((static_cast<size_t>(slot) * a.h_v + h) * D + j) * D;
                        else if (slot >= 0 && tid == 0)
                            report(a.dev_status, GDN_DEV_BAD_SLOT);
                    } else if (a.chunk_states) {
                        const int64_t idx = eoff + (c + 1) / E - 1;
                        if (idx >= 0 && idx < a.chunk_capacity)
                            ep = a.chunk_states + ((static_cast<size_t>(idx) * a.h_v + h) * D + j) * D;
                    }
                }
                float *dp = (c == n_chunks - 1 && dst >= 0)
                                ? a.state + ((static_cast<size_t>(dst) * a.h_v + h) * D + j) * D
                                : nullptr;
#pragma unroll 1
                for (int c0 = hf * kHalf; c0 < (hf + 1) * kHalf; c0 += 32) {
                    uint32_t r[32], p16[16];
                    tc::tmem_ld32(tl + kColS + c0, r);
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        p16[i] = pack_half2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                    tc::tmem_st16(tl + kColS16 + c0 / 2, p16);
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        const float4 v = make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]),
                                                     __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
                        if (ep) __stcg(reinterpret_cast<float4 *>(ep + c0 + i), v);
                        if (dp) __stcg(reinterpret_cast<float4 *>(dp + c0 + i), v);
                    }
                }
            }
            tc::fence_before_sync();
            if (group_any(kBarChain, !okc || *vfail)) {
                failed = true;
                break;
            }
            prev_n = n;
            prev_tok0 = tok0;
        }
        if (!failed && n_chunks > 0 && jv) output(prev_n, prev_tok0, hf);
        if (failed && tid == 0) {
            report(a.dev_status, GDN_DEV_TIMEOUT);
            atomicExch(fail, 1);
        }
        if (tid == 0) {  // every MMA this thread issued has finished before TMEM is released
            tc::mma_commit(bars + kBarDrainC);
            drain_bar(bars + kBarDrainC, 0);
        }
    } else {
        // ============================= prep group ==============================
        // Thread (p, hf): TMEM lane / product row p, half hf of the row's columns.
        const int pid = tid - kGroup;  // 0..255
        const int p = pid & 127, hf = pid >> 7;
        bool failed = false;
        int c_done = 0;                          // chunks whose loads the loop consumed
        int qk_issued = -1, v_issued = -1;       // highest chunk whose copies this thread issued (pid 0, 64)
        constexpr uint32_t kQKTx = 2u * kKB * 8192u, kVTx = kKB * 8192u;
        // g and beta of a chunk, tokens 2l and 2l + 1 in lane l of warp 10 (zeros
        // past the sequence end), loaded a chunk ahead.
        float gv0 = 0.f, gv1 = 0.f, bv0 = 0.f, bv1 = 0.f;
        auto load_gb = [&](int cc) {
            if (warp == 10) {
                const int nn = min(kChunk, Lseq - cc * kChunk), l = pid & 31;
                const size_t gi = static_cast<size_t>(t0 + cc * kChunk + 2 * l) * a.h_v + h;
                gv0 = 2 * l < nn ? a.g[gi] : 0.f;
                bv0 = 2 * l < nn ? a.beta[gi] : 0.f;
                gv1 = 2 * l + 1 < nn ? a.g[gi + a.h_v] : 0.f;
                bv1 = 2 * l + 1 < nn ? a.beta[gi + a.h_v] : 0.f;
            }
        };
        auto issue_qk = [&](int cc) {  // q and k of chunk cc into slot cc % 3
            uint8_t *tile = sQK(cc % 3);
            uint64_t *tb = bars + kBarTmaQK + cc % 3;
            mbar_expect_tx(tb, kQKTx);
#pragma unroll
            for (int kb = 0; kb < kKB; ++kb) {
                tma_load_2d(tile + kb * 16384, &L.tm_q, kh * D + kb * 64, t0 + cc * kChunk, tb);
                tma_load_2d(tile + kb * 16384 + 8192, &L.tm_k, kh * D + kb * 64, t0 + cc * kChunk, tb);
            }
            qk_issued = cc;
        };
        auto issue_v = [&](int cc) {  // v of chunk cc into slot cc & 1
            uint8_t *tile = sV(cc & 1);
            uint64_t *tb = bars + kBarTmaV + (cc & 1);
            mbar_expect_tx(tb, kVTx);
#pragma unroll
            for (int kb = 0; kb < kKB; ++kb) tma_load_2d(tile + kb * 8192, &L.tm_v, h * D + kb * 64, t0 + cc * kChunk, tb);
            v_issued = cc;
        };
        if (n_chunks > 0) {
            if (pid == 0) {
                issue_qk(0);
                issue_v(0);
                if (n_chunks > 1) {
                    issue_qk(1);
                    issue_v(1);
                }
                // the first chunk's Gram (the chain group queues the later ones)
                if (wait_bar(bars + kBarTmaQK, 0, fail)) {
                    tc::fence_after_sync();
                    gram_mma<D>(tbase, sQK(0), bars + kBarGram);
                } else {
                    atomicExch(fail, 1);
                }
            }
            load_gb(0);
        }

        for (int c = 0; c < n_chunks; ++c) {
            const int s = c & 1;
            const int n = min(kChunk, Lseq - c * kChunk);
            uint8_t *qk = sQK(c % 3);
            uint8_t *vt = sV(c & 1);

            // ---- Q2: prefix sum of the decays (the Gram is already running) -----------
            bool ok = true;
            if (warp == 10) {  // inclusive prefix sum of g over the chunk, fixed order
                const int l = pid & 31;
                const float g0 = gv0, g1 = gv1;
                sBeta[2 * l] = bv0;
                sBeta[2 * l + 1] = bv1;
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
                const float e0 = expf(G0), e1 = expf(G1);
                sGl[2 * l] = G0 * 1.4426950408889634f;
                sGl[2 * l + 1] = G1 * 1.4426950408889634f;
                sGam[2 * l] = e0;
                sGam[2 * l + 1] = e1;
                sBG[2 * l] = bv0 * e0;
                sBG[2 * l + 1] = bv1 * e1;
                sDec(s)[2 * l] = expf(Gc - G0);
                sDec(s)[2 * l + 1] = expf(Gc - G1);
                if (l == 31) sGc[s] = e1;
                __syncwarp();
                if (l == 0) mbar_arrive(bars + kBarGamReady);
                if (c + 1 < n_chunks) load_gb(c + 1);
            }
            if (group_any(kBarPrep, !ok || *vfail)) {
                failed = true;
                break;
            }

            // ---- Q3: P~ rows (lanes 0..63) and A rows (lanes 64..127), columns 32 hf.. --
            // Rows 0..31 x columns 32..63 are masked (warp-uniform): P~ gets zeros,
            // the upper triangle of A is never read.
            const bool okg = __all_sync(0xffffffffu, wait_bar(bars + kBarGram, c & 1, fail));
            tc::fence_after_sync();
            if (!okg) {
                // the barrier below ends the loop
            } else if (hf == 1 && (p & 32) == 0) {
                if (p < 64) {
                    const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int q = 4; q < 8; ++q)
                        *reinterpret_cast<uint4 *>(sP(s) + tc::sw128_chunk_offset(p & 63, q, 64)) = z;
                }
            } else {
                // exp(G_r - G_c) f = exp2(Gl_r + log2 f - Gl_c) with Gl = G log2(e);
                // f = beta_r (A rows) is folded into the exponent when positive.
                // Only the warps on a diagonal 32 x 32 block apply the mask.
                uint32_t x[32];
                tc::tmem_ld32(tl + kColGram + 32 * hf, x);
                const int r = p & 63;
                const bool isA = p >= 64;
                const float br = isA ? sBeta[r] : 1.f;
                const bool fold = br > 0.f;
                const float Er = sGl[r] + (fold ? __log2f(br) : 0.f);
                const float post = isA ? (fold ? 1.f : br) : a.scale;
                const bool diag_blk = (hf == 0) == ((p & 32) == 0);  // warp-uniform
                const int lim = isA ? r - 1 : r;                      // A: s < t, P~: s <= t
#pragma unroll
                for (int q4 = 0; q4 < 32; q4 += 4) {
                    const int q0 = 32 * hf + q4;
                    const float4 g4 = *reinterpret_cast<const float4 *>(sGl + q0);
                    const float gg[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        float y = exp2f_approx(Er - gg[u]) * __uint_as_float(x[q4 + u]);
                        if (diag_blk && q0 + u > lim) y = 0.f;
                        x[q4 + u] = __float_as_uint(y);
                    }
                }
                if (post != 1.f) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[i] = __float_as_uint(post * __uint_as_float(x[i]));
                }
                if (p < 64) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 v;
                        v.x = pack_half2(__uint_as_float(x[8 * q + 0]), __uint_as_float(x[8 * q + 1]));
                        v.y = pack_half2(__uint_as_float(x[8 * q + 2]), __uint_as_float(x[8 * q + 3]));
                        v.z = pack_half2(__uint_as_float(x[8 * q + 4]), __uint_as_float(x[8 * q + 5]));
                        v.w = pack_half2(__uint_as_float(x[8 * q + 6]), __uint_as_float(x[8 * q + 7]));
                        *reinterpret_cast<uint4 *>(sP(s) + tc::sw128_chunk_offset(r, 4 * hf + q, 64)) = v;
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 32; q += 4)
                        *reinterpret_cast<float4 *>(sM + r * kLdM + 32 * hf + q) =
                            make_float4(__uint_as_float(x[q]), __uint_as_float(x[q + 1]), __uint_as_float(x[q + 2]),
                                        __uint_as_float(x[q + 3]));
                    if (r >= 32 && hf == 0) store_row32_f16(sL2A1, r - 32, x, 1.f, true);  // A_B, fp16
                }
            }
            tc::fence_proxy_async_smem();
            tc::fence_before_sync();
            if (group_any(kBarPrep, !okg || *vfail)) {
                failed = true;
                break;
            }
            if (pid == 0) mbar_arrive(bars + kBarGramFree);  // the chain may issue the next Gram

            // ---- Q4: diagonal blocks (warps 8, 9) and level 1 (warps 8, 9, 12, 13) -------
            bool okv = true;
            if (pid == 64 && c >= 1) {
                // T'' and the v slot of chunk c - 1 are free once the chain's U'^T
                // product of that chunk is done (long before this point): the v
                // copies of chunk c + 1 go there, a whole chunk ahead (issued by
                // warp 10, idle in this phase).
                okv = wait_bar(bars + kBarTFree, (c - 1) & 1, fail);
                if (okv && c + 1 < n_chunks) issue_v(c + 1);
            }
            if (pid < 64) {
                float xd[16];
                invert_diag_solve(sM, pid, xd);
                __syncwarp();
                invert_diag_store(sM, pid, xd);
                // level 1 in two halves: this warp and warp 12 (or 13)
                if (pid < 32) level1_half<1>(sM, sWb, pid & 31, 0, kBarPairL1);
                else level1_half<3>(sM, sWb, pid & 31, 0, kBarPairL1 + 1);
                // Level-2 operands: T_top (rows 0..31, cols 0..31) as MN-major B
                // (warp 8), T_bot (rows 32..63, cols 32..63) as K-major A (warp 9);
                // the blocks above the diagonal blocks are zero.
                const int r = pid & 31;
                const int rb = pid < 32 ? 0 : 32;
                uint32_t x[32];
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    x[i] = (i >= 16 && r < 16) ? 0u : __float_as_uint(sM[(rb + r) * kLdM + rb + i]);
                store_row32_f16(pid < 32 ? sL2B1 : sL2A2, r, x, 1.f, pid >= 32);
            } else if (pid >= 128 && pid < 192) {  // warps 12, 13: the other half of level 1
                if (pid < 160) level1_half<1>(sM, sWb, pid & 31, 1, kBarPairL1);
                else level1_half<3>(sM, sWb, pid & 31, 1, kBarPairL1 + 1);
            }
            tc::fence_proxy_async_smem();
            tc::fence_before_sync();
            if (group_any(kBarPrep, !okv || *vfail)) {
                failed = true;
                break;
            }
            c_done = c;  // this chunk's copies have all been waited for

            // ---- Q5: level 2 on the tensor cores (warp 8) || T'', -T''' of the rest ---
            bool okl = true;
            if (pid < 32) {
                // X = A_B T_top, then T_B = T_bot (-X): lanes 0..31 of the prep columns.
                if (pid == 0) {
                    tc::fence_after_sync();
                    const uint64_t dA = tc::desc_k_sw128(tc::smem_u32(sL2A1));
                    const uint64_t dB = tc::desc_mn_sw128(tc::smem_u32(sL2B1), 0);
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
                        tc::mma_f16(tbase + kColPrep, dA + kk * 2, dB + kk * (2048 >> 4),
                                    tc::idesc_f16_f32acc(128, 32) | tc::kIdescBmn, kk > 0);
                    tc::mma_commit(bars + kBarL2);
                }
                __syncwarp();
                okl = __all_sync(0xffffffffu, wait_bar(bars + kBarL2, 0, fail));
                tc::fence_after_sync();
                uint32_t x[32];
                if (okl) {
                    tc::tmem_ld32(tl + kColPrep, x);
                    store_row32_f16(sL2B2, pid, x, -1.f, false);
                }
                tc::fence_proxy_async_smem();
                tc::fence_before_sync();
                __syncwarp();
                if (pid == 0 && okl) {
                    tc::fence_after_sync();
                    const uint64_t dA = tc::desc_k_sw128(tc::smem_u32(sL2A2));
                    const uint64_t dB = tc::desc_mn_sw128(tc::smem_u32(sL2B2), 0);
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
                        tc::mma_f16(tbase + kColPrep + 32, dA + kk * 2, dB + kk * (2048 >> 4),
                                    tc::idesc_f16_f32acc(128, 32) | tc::kIdescBmn, kk > 0);
                    tc::mma_commit(bars + kBarL2);
                }
                __syncwarp();
                okl = okl && __all_sync(0xffffffffu, wait_bar(bars + kBarL2, 1, fail));
                tc::fence_after_sync();
                if (okl) {  // T_B: row 32 + pid, columns 0..31
                    tc::tmem_ld32(tl + kColPrep + 32, x);
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        float v[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(x[16 * q + i]);
                        store_t_segment(sTpp, sTppp, 32 + pid, q, v, sBeta, sBG);
                    }
                }
            } else if (pid >= 64) {
                // 16-column row segments of T (all but rows 32..63 x cols 0..31).
                const int g = pid - 64;
                const int t = g < 128 ? (g >> 2) : 32 + ((g - 128) >> 1);
                const int q = g < 128 ? (g & 3) : 2 + ((g - 128) & 1);
                float v[16];
                if (q > (t >> 4)) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = 0.f;
                } else {
#pragma unroll
                    for (int i = 0; i < 16; i += 4) {
                        const float4 m4 = *reinterpret_cast<const float4 *>(sM + t * kLdM + 16 * q + i);
                        v[i] = m4.x;
                        v[i + 1] = m4.y;
                        v[i + 2] = m4.z;
                        v[i + 3] = m4.w;
                    }
                }
                store_t_segment(sTpp, sTppp, t, q, v, sBeta, sBG);
            }
            tc::fence_proxy_async_smem();
            tc::fence_before_sync();
            if (group_any(kBarPrep, !okl || *vfail)) {
                failed = true;
                break;
            }
            if (pid == 0) mbar_arrive(bars + kBarUReady);  // T'' and v of chunk c ready

            // ---- Q6: -W^T = K^T (-T''')^T -> fp16 tile --------------------------------
            if (pid == 0) {
                ok = ((c == 0) || wait_bar(bars + kBarWFree, (c - 1) & 1, fail)) &&
                     wait_bar(bars + kBarConvDone, c & 1, fail);  // k of chunk c in fp16
                if (ok) {
                    tc::fence_after_sync();
                    const uint64_t dK = tc::desc_mn_sw128(tc::smem_u32(qk + 8192), kLboK);
                    const uint64_t dT = tc::desc_k_sw128(tc::smem_u32(sTppp));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc::mma_f16(tbase + kColPrep, dK + kk * (2048 >> 4), dT + kk * 2,
                                    tc::idesc_f16_f32acc(128, 64) | tc::kIdescAmn, kk > 0);
                    tc::mma_commit(bars + kBarW);
                } else {
                    atomicExch(fail, 1);
                }
            }
            __syncwarp();
            const bool okw = __all_sync(0xffffffffu, wait_bar(bars + kBarW, c & 1, fail));
            tc::fence_after_sync();
            if (okw && p < D) {  // row i = p of the MN-major -W^T tile, tokens 32 hf ..
                uint32_t x[32];
                tc::tmem_ld32(tl + kColPrep + 32 * hf, x);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 v;
                    v.x = pack_half2(__uint_as_float(x[8 * q + 0]), __uint_as_float(x[8 * q + 1]));
                    v.y = pack_half2(__uint_as_float(x[8 * q + 2]), __uint_as_float(x[8 * q + 3]));
                    v.z = pack_half2(__uint_as_float(x[8 * q + 4]), __uint_as_float(x[8 * q + 5]));
                    v.w = pack_half2(__uint_as_float(x[8 * q + 6]), __uint_as_float(x[8 * q + 7]));
                    *reinterpret_cast<uint4 *>(sWT + mn_chunk_offset(p, 4 * hf + q)) = v;
                }
            }
            tc::fence_proxy_async_smem();
            tc::fence_before_sync();
            if (group_any(kBarPrep, !okw || *vfail)) {
                failed = true;
                break;
            }
            // ---- hand over: q/k copies of chunk c + 2 into the slot of chunk c - 1 ----
            if (pid == 0) {
                mbar_arrive(bars + kBarReady + s);
                bool okq = true;
                // The chain is done with chunk c - 1 (q/k slot, P~ and decay stage)
                // before the next chunk's preparation reuses them.
                if (okq && c >= 1) okq = wait_bar(bars + kBarQKFree, (c - 1) & 1, fail);
                if (okq && c + 2 < n_chunks) issue_qk(c + 2);
                if (!okq) atomicExch(fail, 1);
            }
            c_done = c + 1;
        }
        if (failed && pid == 0) {
            report(a.dev_status, GDN_DEV_TIMEOUT);
            atomicExch(fail, 1);
        }
        if (pid == 0) {  // drain: this thread's MMAs, then every copy it issued that the loop did not consume
            tc::mma_commit(bars + kBarDrainP);
            drain_bar(bars + kBarDrainP, 0);
            for (int cc = c_done; cc <= qk_issued; ++cc) drain_bar(bars + kBarTmaQK + cc % 3, (cc / 3) & 1);
            for (int cc = c_done; cc <= v_issued; ++cc) drain_bar(bars + kBarTmaV + (cc & 1), (cc / 2) & 1);
        }
        if (pid == 64)  // the v copies this thread issued
            for (int cc = c_done; cc <= v_issued; ++cc) drain_bar(bars + kBarTmaV + (cc & 1), (cc / 2) & 1);
    }

    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tbase, kTmemCols);
}

// Dynamic shared memory is opted into once per device and head dim.
template <int D>
cudaError_t launch_d(const PrefillLaunch &L, cudaStream_t stream) {
    static int set[kMaxDevices] = {};
    const uint32_t smem = Smem<D>::kAlloc;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices || !__atomic_load_n(&set[dev], __ATOMIC_ACQUIRE)) {
        e = cudaFuncSetAttribute(prefill_chain_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kMaxDevices) __atomic_store_n(&set[dev], 1, __ATOMIC_RELEASE);
    }
    prefill_chain_kernel<D><<<L.a.num_seqs * L.a.h_v, kThreads, smem, stream>>>(L);
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
    PrefillLaunch L;
    L.a = a;
    if (a.total_tokens > 0 &&
        (!encode_rows(&L.tm_q, a.q, a.total_tokens, static_cast<uint64_t>(a.h_k) * d) ||
         !encode_rows(&L.tm_k, a.k, a.total_tokens, static_cast<uint64_t>(a.h_k) * d) ||
         !encode_rows(&L.tm_v, a.v, a.total_tokens, static_cast<uint64_t>(a.h_v) * d)))
        return cudaErrorNotSupported;
    // Longest sequences first, so the longest chains start in the first wave
    // (stable: equal lengths keep their order); beyond kMaxOrder sequences the
    // rest keep their order.
    L.n_order = a.num_seqs < kMaxOrder ? a.num_seqs : kMaxOrder;
    for (int i = 0; i < L.n_order; ++i) L.order[i] = i;
    std::stable_sort(L.order, L.order + L.n_order, [cu_host](int x, int y) {
        return cu_host[x + 1] - cu_host[x] > cu_host[y + 1] - cu_host[y];
    });
    return d == 128 ? launch_d<128>(L, stream) : launch_d<64>(L, stream);
}

}  // namespace gdn
