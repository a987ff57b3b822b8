// Packed recurrent decode: one token per cached row against its fp32 state,
// and the multi-token form for rows carrying several (speculative) tokens.
//
// vLLM page "Enable batch-invariant mixed decode and prefill for Qwen GDN",
// section "How": cached rows always go through this packed recurrent decode,
// alone or at the front of a mixed batch.
//
// The kernel is bound by HBM: each (row, value head) state S^T [d_v][d_k] fp32
// (64 KiB at d = 128) is read once and written once; q, k, v, g, beta and o
// add about 1.6 %.  Work is split into items of 8 state rows (4 KiB); a
// persistent grid of warps walks the items with a grid stride, so each warp
// has its item's loads in flight at once and the grid fills every SM
// regardless of the row count.  State stores are streaming (.cs): the block
// is not read again within the launch.  Measured, 8-row items with
// streaming stores move the most bytes per second (16-row items or .cg
// stores are ~3 % slower).  Arithmetic per state row is in row_update.cuh.
#include "row_update.cuh"

namespace gdn {
namespace {

constexpr int kDecodeThreads = 128;  // measured best: 128 > 64 > 256 > 512 threads per block
constexpr int kMultiThreads = 256;
constexpr int kRowsPerGroup = 4;  // rows of S^T per warp-wide access (lane octets)
constexpr int kGroupsPerItem = 2;
constexpr int kRowsPerItem = kRowsPerGroup * kGroupsPerItem;  // 8

// Five blocks per SM (96 registers, no spills) measured best: 20 warps per SM.
template <int D, bool kRaw>
__global__ void __launch_bounds__(kDecodeThreads, 5)
decode_kernel(const DecodeArgs a) {
    constexpr int V4 = D / 32;                   // float4 per lane per row
    constexpr int kItemsPerHead = D / kRowsPerItem;
    const int lane = threadIdx.x & 31;
    const int sub = lane >> 3;
    const int l8 = lane & 7;
    const int64_t n_items = static_cast<int64_t>(a.num_rows) * a.h_v * kItemsPerHead;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int group = a.h_v / a.h_k;

    for (int64_t it = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
         it < n_items; it += nwarps) {
        const int blk = static_cast<int>(it % kItemsPerHead);
        const int64_t rh = it / kItemsPerHead;
        const int h = static_cast<int>(rh % a.h_v);
        const int r = static_cast<int>(rh / a.h_v);
        const int row0 = blk * kRowsPerItem;
        uint16_t *orow = a.o + (static_cast<size_t>(r) * a.h_v + h) * D;

        const int src = a.src_slot[r];
        const int dst = a.dst_slot ? a.dst_slot[r] : src;
        if (src < 0 || src >= a.num_slots || dst < 0 || dst >= a.num_slots) {
            if (src >= 0) report(a.dev_status, GDN_DEV_BAD_SLOT);
            if (lane < kRowsPerItem) orow[row0 + lane] = 0;
            continue;
        }
        const float *sp = a.state + (static_cast<size_t>(src) * a.h_v + h) * D * D;
        float *dp = a.state + (static_cast<size_t>(dst) * a.h_v + h) * D * D;

        float4 s[kGroupsPerItem][V4];
#pragma unroll
        for (int i = 0; i < kGroupsPerItem; ++i) {
            const int j = row0 + i * kRowsPerGroup + sub;
#pragma unroll
            for (int m = 0; m < V4; ++m)
                s[i][m] = ld_state4(sp + static_cast<size_t>(j) * D + 4 * (l8 + 8 * m));
        }
        const int kh = h / group;
        float kk[V4 * 4], qq[V4 * 4];
        load_bf16_slice<V4>(a.k + (static_cast<size_t>(r) * a.h_k + kh) * D, l8, kk);
        load_bf16_slice<V4>(a.q + (static_cast<size_t>(r) * a.h_k + kh) * D, l8, qq);
        const size_t gh = static_cast<size_t>(r) * a.h_v + h;
        float g, beta;
        if constexpr (kRaw) {  // fused input preparation
            normalize_bf16<V4>(kk, a.eps);
            normalize_bf16<V4>(qq, a.eps);
            gate_inputs(a.a_raw[gh], a.b_raw[gh], a.A_log[h], a.dt_bias[h], g, beta);
        } else {
            g = a.g[gh];
            beta = a.beta[gh];
        }
        const float alpha = expf(g);
        const float kq = octet_dot<V4>(kk, qq);
        const uint16_t *vrow = a.v + gh * D;

#pragma unroll
        for (int i = 0; i < kGroupsPerItem; ++i) {
            const int j = row0 + i * kRowsPerGroup + sub;
            const float vj = bf16_bits_to_float(vrow[j]);
            const float oj = update_row<V4>(s[i], kk, qq, alpha, beta, vj, kq, a.scale);
#pragma unroll
            for (int m = 0; m < V4; ++m)
                __stcs(reinterpret_cast<float4 *>(dp + static_cast<size_t>(j) * D + 4 * (l8 + 8 * m)),
                       s[i][m]);
            if (l8 == 0) orow[j] = float_to_bf16_bits(oj);
        }
    }
}

// Items of the multi-token form: 16 rows, since every token of the row adds
// q, k, v loads and reductions to the item (measured: 8-row items are ~15 %
// slower here, unlike the single-token decode).
constexpr int kMultiGroups = 4;  // update_rows4_scatter takes the four rows of an octet
constexpr int kMultiRows = kRowsPerGroup * kMultiGroups;  // 16

// Multi-token decode (speculative tokens): the item's 16 state rows stay in
// registers across the row's tokens, whose inputs (up to kStageTokens of them)
// are staged in shared memory by asynchronous copies issued before the state
// is loaded; after token t the state is stored at
// dst_slots[r * T + t] when that entry is >= 0 (a snapshot a verifier can
// roll back to), or, with dst_slots == NULL, once after the last token back
// to src_slot[r].  Every step has the packed decode's per-row arithmetic
// (update_row; here the reductions of an item's rows are done together as a
// reduce-scatter of the same sums), so T tokens here equal T packed-decode
// calls bit for bit.
// Per warp, the inputs of up to kStageTokens tokens of its current row are
// staged in shared memory by asynchronous copies issued when the item starts:
// one memory round trip per item instead of one per token.
constexpr int kStageTokens = 8;

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
                 "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
                 "l"(gmem)
                 : "memory");
}

// Stage of decode_multi_kernel, per token.  kF32: k and q as fp32 (the
// copies land as bf16 in the upper half of the same bytes and the warp
// converts them once per token), else k and q as the bf16 rows the copies
// bring; then the item's v (bf16), g and beta.  The fp32 form measured faster
// at 3-4 tokens per row and slower at 1-2 and 8 (its per-item conversion
// round is not overlapped with arithmetic), so the launcher picks it for rows
// of 3 or 4 tokens.
template <int D, bool kF32>
struct MultiStageT {
    static constexpr int kK = 0, kQ = kF32 ? 4 * D : 2 * D;
    static constexpr int kKraw = kF32 ? 4 * D : 0, kQraw = kF32 ? 6 * D : 2 * D;
    static constexpr int kV = kF32 ? 8 * D : 4 * D, kG = kV + 2 * kMultiRows, kB = kG + 16;
    static constexpr int kBytes = kB + 16;
    static constexpr int kBlock = (kMultiThreads / 32) * kStageTokens * kBytes;
};

template <int V4>
__device__ __forceinline__ void load_f32_slice(const float *p, int l8, float (&x)[V4 * 4]) {
#pragma unroll
    for (int m = 0; m < V4; ++m) {
        const float4 w = *reinterpret_cast<const float4 *>(p + 4 * (l8 + 8 * m));
        x[4 * m + 0] = w.x;
        x[4 * m + 1] = w.y;
        x[4 * m + 2] = w.z;
        x[4 * m + 3] = w.w;
    }
}

// Position of a multi-token item, item = (r * h_v + h) * (D / kMultiRows) + b,
// advanced from one of a warp's items to its next by mixed-radix addition
// (no divisions in the loop).
struct ItemPos {
    int b, h, r;
};
struct ItemStep {
    int db, dh, dr;
};
__device__ __forceinline__ ItemPos item_pos(int64_t it, int items_per_head, int h_v) {
    const int64_t rh = it / items_per_head;
    return ItemPos{static_cast<int>(it % items_per_head), static_cast<int>(rh % h_v), static_cast<int>(rh / h_v)};
}
__device__ __forceinline__ ItemPos item_next(ItemPos p, ItemStep s, int items_per_head, int h_v) {
    p.b += s.db;
    const int cb = p.b >= items_per_head;
    p.b -= cb ? items_per_head : 0;
    p.h += s.dh + cb;
    const int ch = p.h >= h_v;
    p.h -= ch ? h_v : 0;
    p.r += s.dr + ch;
    return p;
}

template <int D, bool kF32>
__global__ void __launch_bounds__(kMultiThreads, 2)
decode_multi_kernel(const DecodeMultiArgs a) {
    constexpr int V4 = D / 32;
    constexpr int kItemsPerHead = D / kMultiRows;
    using MS = MultiStageT<D, kF32>;
    extern __shared__ __align__(16) uint8_t multi_smem[];
    const int lane = threadIdx.x & 31;
    const int sub = lane >> 3;
    const int l8 = lane & 7;
    const int T = a.tokens_per_row;
    const int group = a.h_v / a.h_k;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const ItemPos dpos = item_pos(nwarps, kItemsPerHead, a.h_v);
    const ItemStep step{dpos.b, dpos.h, dpos.r};
    // per-token strides of the token-major inputs and outputs
    const size_t kq_stride = static_cast<size_t>(a.h_k) * D, hv_stride = static_cast<size_t>(a.h_v) * D;

    const bool staged = T <= kStageTokens;
    // With several tokens per row and only the final state written, an item's
    // arithmetic outlasts its loads, so the next item's state is fetched into
    // L2 ahead of time (measured: with snapshots, or at one or two tokens, the
    // extra requests only compete with the kernel's own traffic).
    const bool prefetch = a.dst_slots == nullptr && T >= 3;
    uint8_t(*stage)[MS::kBytes] =
        reinterpret_cast<uint8_t(*)[MS::kBytes]>(multi_smem + (threadIdx.x >> 5) * kStageTokens * MS::kBytes);

    ItemPos cur = item_pos((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5, kItemsPerHead, a.h_v);
    for (; cur.r < a.num_rows; cur = item_next(cur, step, kItemsPerHead, a.h_v)) {
        const int h = cur.h, r = cur.r, row0 = cur.b * kMultiRows;
        const int kh = h / group;
        const size_t tok0 = static_cast<size_t>(r) * T;  // the row's first token
        if (staged) {
            // Copies of the item's token inputs into this warp's stage (one
            // commit group): rows of k and q (D / 8 16-byte pieces each), the
            // item's v (kMultiRows / 8 pieces), g and beta.
            __syncwarp();  // the previous item's reads of the stage are done
            if (lane < D / 8) {
                const uint16_t *pk = a.k + (tok0 * a.h_k + kh) * D + 8 * lane;
                const uint16_t *pq = a.q + (tok0 * a.h_k + kh) * D + 8 * lane;
                for (int t = 0; t < T; ++t, pk += kq_stride, pq += kq_stride) {
                    cp_async16(stage[t] + MS::kKraw + 16 * lane, pk);
                    cp_async16(stage[t] + MS::kQraw + 16 * lane, pq);
                }
            } else if (lane < D / 8 + kMultiRows / 8) {
                const int pc = lane - D / 8;
                const uint16_t *pv = a.v + (tok0 * a.h_v + h) * D + row0 + 8 * pc;
                for (int t = 0; t < T; ++t, pv += hv_stride) cp_async16(stage[t] + MS::kV + 16 * pc, pv);
            } else if (lane >= 30) {
                const float *pg = (lane == 30 ? a.g : a.beta) + tok0 * a.h_v + h;
                const int off = lane == 30 ? MS::kG : MS::kB;
                for (int t = 0; t < T; ++t, pg += a.h_v) cp_async4(stage[t] + off, pg);
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        }

        uint16_t *orow = a.o + (tok0 * a.h_v + h) * D;  // token t: + t * hv_stride
        const int src = a.src_slot[r];
        if (src < 0 || src >= a.num_slots) {
            if (src >= 0) report(a.dev_status, GDN_DEV_BAD_SLOT);
            for (int t = 0; t < T; ++t, orow += hv_stride)
                if (lane < kMultiRows) orow[row0 + lane] = 0;
            // the stage is refilled by the next item only after these copies land
            if (staged) asm volatile("cp.async.wait_group 0;" ::: "memory");
            continue;
        }
        const float *sp = a.state + (static_cast<size_t>(src) * a.h_v + h) * D * D;
        float4 s[kMultiGroups][V4];
#pragma unroll
        for (int i = 0; i < kMultiGroups; ++i) {
            const int j = row0 + i * kRowsPerGroup + sub;
#pragma unroll
            for (int m = 0; m < V4; ++m)
                s[i][m] = ld_state4(sp + static_cast<size_t>(j) * D + 4 * (l8 + 8 * m));
        }
        // The next item's state rows (8 KB, contiguous) are requested into L2
        // with one bulk prefetch while this item's tokens run.
        if (prefetch && lane == 0) {
            const ItemPos nx = item_next(cur, step, kItemsPerHead, a.h_v);
            if (nx.r < a.num_rows) {
                const int nsrc = a.src_slot[nx.r];
                if (nsrc >= 0 && nsrc < a.num_slots) {
                    const float *np =
                        a.state + ((static_cast<size_t>(nsrc) * a.h_v + nx.h) * D + nx.b * kMultiRows) * D;
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(np), "r"(kMultiRows * D * 4)
                                 : "memory");
                }
            }
        }
        if (staged) {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
            __syncwarp();
        }
        if (kF32 && staged) {
            // k and q of every token to fp32, in place: lane L reads 8 bf16 of
            // the upper half and, once all lanes have read, writes them as 8 floats
            for (int t = 0; t < T; ++t) {
                uint4 w = make_uint4(0u, 0u, 0u, 0u);
                if (lane < D / 4) w = *reinterpret_cast<const uint4 *>(stage[t] + MS::kKraw + 16 * lane);
                __syncwarp();
                if (lane < D / 4) {
                    float4 *dst = reinterpret_cast<float4 *>(stage[t] + 32 * lane);
                    dst[0] = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                                         __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
                    dst[1] = make_float4(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xffff0000u),
                                         __uint_as_float(w.w << 16), __uint_as_float(w.w & 0xffff0000u));
                }
            }
            __syncwarp();
        }
        // lane l8 of the octet takes v of, and writes o of, row (l8 & 3) * 4 + octet
        const int jo = row0 + (l8 & 3) * kRowsPerGroup + sub;
        for (int t = 0; t < T; ++t, orow += hv_stride) {
            float kk[V4 * 4], qq[V4 * 4];
            float alpha, beta, vj;
            if (staged) {
                if constexpr (kF32) {
                    load_f32_slice<V4>(reinterpret_cast<const float *>(stage[t] + MS::kK), l8, kk);
                    load_f32_slice<V4>(reinterpret_cast<const float *>(stage[t] + MS::kQ), l8, qq);
                } else {
                    load_bf16_slice<V4>(reinterpret_cast<const uint16_t *>(stage[t] + MS::kK), l8, kk);
                    load_bf16_slice<V4>(reinterpret_cast<const uint16_t *>(stage[t] + MS::kQ), l8, qq);
                }
                alpha = expf(*reinterpret_cast<const float *>(stage[t] + MS::kG));
                beta = *reinterpret_cast<const float *>(stage[t] + MS::kB);
                vj = bf16_bits_to_float(reinterpret_cast<const uint16_t *>(stage[t] + MS::kV)[jo - row0]);
            } else {
                const size_t tok = tok0 + t, gh = tok * a.h_v + h;
                load_bf16_slice<V4>(a.k + (tok * a.h_k + kh) * D, l8, kk);
                load_bf16_slice<V4>(a.q + (tok * a.h_k + kh) * D, l8, qq);
                alpha = expf(a.g[gh]);
                beta = a.beta[gh];
                vj = bf16_bits_to_float(a.v[gh * D + jo]);
            }
            const float kq = octet_dot<V4>(kk, qq);
            int dst = -1;
            if (a.dst_slots) {
                dst = a.dst_slots[tok0 + t];
                if (dst >= a.num_slots) {
                    report(a.dev_status, GDN_DEV_BAD_SLOT);
                    dst = -1;
                }
            } else if (t == T - 1) {
                dst = src;
            }
            const float oj = update_rows4_scatter<V4>(s, kk, qq, alpha, beta, vj, kq, a.scale, lane);
            if (dst >= 0) {
                float *dp = a.state + (static_cast<size_t>(dst) * a.h_v + h) * D * D;
#pragma unroll
                for (int i = 0; i < kMultiGroups; ++i) {
                    const int j = row0 + i * kRowsPerGroup + sub;
#pragma unroll
                    for (int m = 0; m < V4; ++m)
                        __stcs(reinterpret_cast<float4 *>(dp + static_cast<size_t>(j) * D + 4 * (l8 + 8 * m)),
                               s[i][m]);
                }
            }
            if (l8 >= 4) orow[jo] = float_to_bf16_bits(oj);
        }
    }
}

// Multi-token decode for rows of at most kPfTokens tokens: as decode_multi_kernel,
// but each warp also holds its next item in shared memory: while the tokens of
// the current item run from registers, the next item's 16 state rows (8 KB) and
// token inputs are already being copied into the warp's buffers by cp.async, so
// an item starts with shared-memory loads instead of a memory round trip.  The
// token inputs are double-buffered; the state buffer is single: each lane copies
// into it only the pieces it reads back itself, and only after those reads have
// returned their data.
constexpr int kPfTokens = 4;
template <int D>
struct MultiPf {
    using MS = MultiStageT<D, false>;
    static constexpr int kState = kMultiRows * D * 4;   // one item's state rows, fp32
    static constexpr int kStage = kPfTokens * MS::kBytes;
    static constexpr int kWarp = kState + 2 * kStage;   // per warp
    static constexpr int kBlock = (kMultiThreads / 32) * kWarp;
};

template <int D>
__global__ void __launch_bounds__(kMultiThreads, 2)
decode_multi_pf_kernel(const DecodeMultiArgs a) {
    constexpr int V4 = D / 32;
    constexpr int kItemsPerHead = D / kMultiRows;
    using MS = MultiStageT<D, false>;
    using PF = MultiPf<D>;
    extern __shared__ __align__(128) uint8_t pf_smem[];
    const int lane = threadIdx.x & 31;
    const int sub = lane >> 3;
    const int l8 = lane & 7;
    const int T = a.tokens_per_row;
    const int group = a.h_v / a.h_k;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const ItemPos dpos = item_pos(nwarps, kItemsPerHead, a.h_v);
    const ItemStep step{dpos.b, dpos.h, dpos.r};
    const size_t kq_stride = static_cast<size_t>(a.h_k) * D, hv_stride = static_cast<size_t>(a.h_v) * D;
    uint8_t *wbuf = pf_smem + (threadIdx.x >> 5) * PF::kWarp;
    uint8_t *sstate = wbuf;

    // Copies of item p (one commit group): the lane's own state pieces (rows
    // 4 i + sub, float4 columns l8 + 8 m) and the item's token inputs.
    auto issue = [&](ItemPos p, uint8_t *stage) {
        const int row0_ = p.b * kMultiRows, kh_ = p.h / group;
        const size_t tok0_ = static_cast<size_t>(p.r) * T;
        const int src_ = a.src_slot[p.r];
        if (src_ >= 0 && src_ < a.num_slots) {
            const float *sp = a.state + ((static_cast<size_t>(src_) * a.h_v + p.h) * D + row0_) * D;
#pragma unroll
            for (int i = 0; i < kMultiGroups; ++i) {
#pragma unroll
                for (int m = 0; m < V4; ++m) {
                    const int off = (i * kRowsPerGroup + sub) * D + 4 * (l8 + 8 * m);
                    cp_async16(sstate + 4 * off, sp + off);
                }
            }
        }
        if (lane < D / 8) {
            const uint16_t *pk = a.k + (tok0_ * a.h_k + kh_) * D + 8 * lane;
            const uint16_t *pq = a.q + (tok0_ * a.h_k + kh_) * D + 8 * lane;
            for (int t = 0; t < T; ++t, pk += kq_stride, pq += kq_stride) {
                cp_async16(stage + t * MS::kBytes + MS::kK + 16 * lane, pk);
                cp_async16(stage + t * MS::kBytes + MS::kQ + 16 * lane, pq);
            }
        } else if (lane < D / 8 + kMultiRows / 8) {
            const int pc = lane - D / 8;
            const uint16_t *pv = a.v + (tok0_ * a.h_v + p.h) * D + row0_ + 8 * pc;
            for (int t = 0; t < T; ++t, pv += hv_stride) cp_async16(stage + t * MS::kBytes + MS::kV + 16 * pc, pv);
        } else if (lane >= 30) {
            const float *pg = (lane == 30 ? a.g : a.beta) + tok0_ * a.h_v + p.h;
            const int off = lane == 30 ? MS::kG : MS::kB;
            for (int t = 0; t < T; ++t, pg += a.h_v) cp_async4(stage + t * MS::kBytes + off, pg);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    ItemPos cur = item_pos((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5, kItemsPerHead, a.h_v);
    if (cur.r < a.num_rows) issue(cur, wbuf + PF::kState);
    int buf = 0;
    for (; cur.r < a.num_rows; buf ^= 1) {
        uint8_t *stage_buf = wbuf + PF::kState + buf * PF::kStage;
        asm volatile("cp.async.wait_group 0;" ::: "memory");  // this item's copies have landed
        __syncwarp();
        const int h = cur.h, r = cur.r, row0 = cur.b * kMultiRows;
        const size_t tok0 = static_cast<size_t>(r) * T;
        const int src = a.src_slot[r];
        const bool valid = src >= 0 && src < a.num_slots;
        float4 s[kMultiGroups][V4];
        if (valid) {
#pragma unroll
            for (int i = 0; i < kMultiGroups; ++i) {
#pragma unroll
                for (int m = 0; m < V4; ++m) {
                    s[i][m] = *reinterpret_cast<const float4 *>(
                        sstate + 4 * ((i * kRowsPerGroup + sub) * D + 4 * (l8 + 8 * m)));
                    // the read has returned its data before the next item's copy
                    // into the same piece is issued below
                    asm volatile("" ::"f"(s[i][m].x), "f"(s[i][m].y), "f"(s[i][m].z), "f"(s[i][m].w) : "memory");
                }
            }
        }
        // The next item's copies: its state into the state buffer (this lane's
        // pieces, already read above), its token inputs into the other stage.
        const ItemPos nx = item_next(cur, step, kItemsPerHead, a.h_v);
        if (nx.r < a.num_rows) issue(nx, wbuf + PF::kState + (buf ^ 1) * PF::kStage);
        uint16_t *orow = a.o + (tok0 * a.h_v + h) * D;  // token t: + t * hv_stride
        if (!valid) {
            if (src >= 0) report(a.dev_status, GDN_DEV_BAD_SLOT);
            for (int t = 0; t < T; ++t, orow += hv_stride)
                if (lane < kMultiRows) orow[row0 + lane] = 0;
        } else {
            for (int t = 0; t < T; ++t, orow += hv_stride) {
                float kk[V4 * 4], qq[V4 * 4];
                const uint8_t *st = stage_buf + t * MS::kBytes;
                load_bf16_slice<V4>(reinterpret_cast<const uint16_t *>(st + MS::kK), l8, kk);
                load_bf16_slice<V4>(reinterpret_cast<const uint16_t *>(st + MS::kQ), l8, qq);
                const float alpha = expf(*reinterpret_cast<const float *>(st + MS::kG));
                const float beta = *reinterpret_cast<const float *>(st + MS::kB);
                const uint16_t *vrow = reinterpret_cast<const uint16_t *>(st + MS::kV) - row0;
                const float kq = octet_dot<V4>(kk, qq);
                int dst = -1;
                if (a.dst_slots) {
                    dst = a.dst_slots[tok0 + t];
                    if (dst >= a.num_slots) {
                        report(a.dev_status, GDN_DEV_BAD_SLOT);
                        dst = -1;
                    }
                } else if (t == T - 1) {
                    dst = src;
                }
                float *dp = dst >= 0 ? a.state + (static_cast<size_t>(dst) * a.h_v + h) * D * D : nullptr;
#pragma unroll
                for (int i = 0; i < kMultiGroups; ++i) {
                    const int j = row0 + i * kRowsPerGroup + sub;
                    const float vj = bf16_bits_to_float(vrow[j]);
                    const float oj = update_row<V4>(s[i], kk, qq, alpha, beta, vj, kq, a.scale);
                    if (dp) {
#pragma unroll
                        for (int m = 0; m < V4; ++m)
                            __stcs(reinterpret_cast<float4 *>(dp + static_cast<size_t>(j) * D + 4 * (l8 + 8 * m)),
                                   s[i][m]);
                    }
                    if (l8 == 0) orow[j] = float_to_bf16_bits(oj);
                }
            }
        }
        __syncwarp();  // every lane is done with this stage before it is refilled
        cur = nx;
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");  // nothing in flight at exit
}

template <int D, bool kF32>
cudaError_t launch_multi_form(const DecodeMultiArgs &a, int dev, int sms, int64_t need, cudaStream_t stream) {
    static int occ[kMaxDevices] = {}, set[kMaxDevices] = {};
    constexpr int smem = MultiStageT<D, kF32>::kBlock;
    if (dev < 0 || dev >= kMaxDevices || !__atomic_load_n(&set[dev], __ATOMIC_ACQUIRE)) {
        const cudaError_t e =
            cudaFuncSetAttribute(decode_multi_kernel<D, kF32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kMaxDevices) __atomic_store_n(&set[dev], 1, __ATOMIC_RELEASE);
    }
    const int per_sm = blocks_per_sm(decode_multi_kernel<D, kF32>, kMultiThreads, dev, occ, smem);
    const int64_t cap = static_cast<int64_t>(sms) * (per_sm > 0 ? per_sm : 1);
    const int grid = static_cast<int>(need < cap ? need : cap);
    decode_multi_kernel<D, kF32><<<grid, kMultiThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_decode_multi_d(const DecodeMultiArgs &a, cudaStream_t stream) {
    int dev = 0, sms = 0;
    if (!current_device(&dev, &sms)) return cudaErrorInvalidDevice;
    const int64_t items = static_cast<int64_t>(a.num_rows) * a.h_v * (D / kMultiRows);
    const int64_t need = (items + (kMultiThreads / 32) - 1) / (kMultiThreads / 32);
    if (a.dst_slots && a.tokens_per_row <= kPfTokens) {  // snapshots: next item prefetched into shared memory
        static int occ_pf[kMaxDevices] = {}, set[kMaxDevices] = {};
        constexpr int smem = MultiPf<D>::kBlock;
        if (dev < 0 || dev >= kMaxDevices || !__atomic_load_n(&set[dev], __ATOMIC_ACQUIRE)) {
            const cudaError_t e =
                cudaFuncSetAttribute(decode_multi_pf_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < kMaxDevices) __atomic_store_n(&set[dev], 1, __ATOMIC_RELEASE);
        }
        const int per_sm = blocks_per_sm(decode_multi_pf_kernel<D>, kMultiThreads, dev, occ_pf, smem);
        const int64_t cap = static_cast<int64_t>(sms) * (per_sm > 0 ? per_sm : 1);
        const int grid = static_cast<int>(need < cap ? need : cap);
        decode_multi_pf_kernel<D><<<grid, kMultiThreads, smem, stream>>>(a);
        return cudaGetLastError();
    }
    if (a.tokens_per_row >= 3 && a.tokens_per_row <= 4) return launch_multi_form<D, true>(a, dev, sms, need, stream);
    return launch_multi_form<D, false>(a, dev, sms, need, stream);
}

template <int D, bool kRaw>
cudaError_t launch_decode_d(const DecodeArgs &a, cudaStream_t stream) {
    static int occ[kMaxDevices] = {};
    int dev = 0, sms = 0;
    if (!current_device(&dev, &sms)) return cudaErrorInvalidDevice;
    const int per_sm = blocks_per_sm(decode_kernel<D, kRaw>, kDecodeThreads, dev, occ);
    const int64_t items = static_cast<int64_t>(a.num_rows) * a.h_v * (D / kRowsPerItem);
    const int64_t need = (items + (kDecodeThreads / 32) - 1) / (kDecodeThreads / 32);
    const int64_t cap = static_cast<int64_t>(sms) * (per_sm > 0 ? per_sm : 1);
    const int grid = static_cast<int>(need < cap ? need : cap);
    decode_kernel<D, kRaw><<<grid, kDecodeThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, int d, cudaStream_t stream) {
    if (a.num_rows == 0) return cudaSuccess;
    if (a.a_raw) return d == 128 ? launch_decode_d<128, true>(a, stream) : launch_decode_d<64, true>(a, stream);
    return d == 128 ? launch_decode_d<128, false>(a, stream) : launch_decode_d<64, false>(a, stream);
}

cudaError_t launch_decode_multi(const DecodeMultiArgs &a, int d, cudaStream_t stream) {
    if (a.num_rows == 0 || a.tokens_per_row == 0) return cudaSuccess;
    return d == 128 ? launch_decode_multi_d<128>(a, stream) : launch_decode_multi_d<64>(a, stream);
}

}  // namespace gdn
