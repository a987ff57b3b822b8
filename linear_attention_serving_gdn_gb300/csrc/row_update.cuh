// One recurrent step on rows of S^T, held in registers by lane octets.
//
// Layout: a row j of S^T (column j of S, d_k floats) is spread over the 8
// lanes of an aligned lane octet; lane l8 holds the float4s at columns
// 4*(l8 + 8*m), m = 0..V4-1, so one warp-wide float4 access touches 4 rows x
// 128 contiguous bytes.  Per row j, with u the rank-one update of the gated
// delta rule (Gated DeltaNet, Yang, Kautz, Hatamizadeh, ICLR 2025):
//
//     a_j  = sum_i S_ij k_i,   b_j = sum_i S_ij q_i
//     u_j  = beta (v_j - alpha a_j)
//     S'_ij = alpha S_ij + k_i u_j                  (= alpha S - beta k k^T(alpha S) + beta k v^T)
//     o_j  = scale (alpha b_j + u_j (k . q))        (= scale (S'^T q)_j)
//
// Columns j are independent, so any set of rows can be processed by any warp
// and the result of a row never depends on which other rows share the launch.
#pragma once

#include "gdn_internal.cuh"

namespace gdn {

// 16-byte state load, L2-only caching, with a 256-byte L2 fetch hint (the
// lane octet's next segment of the same row is then an L2 hit).
__device__ __forceinline__ float4 ld_state4(const float *p) {
    float4 v;
    asm volatile("ld.global.cg.L2::256B.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

template <int V4>
__device__ __forceinline__ void load_bf16_slice(const uint16_t *p, int l8, float (&x)[V4 * 4]) {
#pragma unroll
    for (int m = 0; m < V4; ++m) {
        const uint2 w = *reinterpret_cast<const uint2 *>(p + 4 * (l8 + 8 * m));
        x[4 * m + 0] = __uint_as_float(w.x << 16);
        x[4 * m + 1] = __uint_as_float(w.x & 0xffff0000u);
        x[4 * m + 2] = __uint_as_float(w.y << 16);
        x[4 * m + 3] = __uint_as_float(w.y & 0xffff0000u);
    }
}

template <int V4>
__device__ __forceinline__ void store_bf16_slice(uint16_t *p, int l8, const float (&x)[V4 * 4]) {
#pragma unroll
    for (int m = 0; m < V4; ++m) {
        uint2 w;
        w.x = static_cast<uint32_t>(float_to_bf16_bits(x[4 * m + 0])) |
              (static_cast<uint32_t>(float_to_bf16_bits(x[4 * m + 1])) << 16);
        w.y = static_cast<uint32_t>(float_to_bf16_bits(x[4 * m + 2])) |
              (static_cast<uint32_t>(float_to_bf16_bits(x[4 * m + 3])) << 16);
        *reinterpret_cast<uint2 *>(p + 4 * (l8 + 8 * m)) = w;
    }
}

// Input preparation of the layer (the pages give no formula; the reading is
// the Gated DeltaNet layer's): per (token, key head)
//     x_hat = x / sqrt(sum x^2 + eps), rounded to bf16,
// and per (token, value head)
//     g = -exp(A_log) softplus(a + dt_bias),  beta = sigmoid(b).
// The sum of squares has one fixed order (each lane of the octet over its
// slice, then the xor butterfly) and every operation is explicitly rounded,
// so the standalone preparation kernel and the fused decode produce the
// same bits.
template <int V4>
__device__ __forceinline__ void normalize_bf16(float (&x)[V4 * 4], float eps) {
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < V4 * 4; ++e) acc = __fmaf_rn(x[e], x[e], acc);
    const float inv = rsqrtf(__fadd_rn(octet_sum(acc), eps));
#pragma unroll
    for (int e = 0; e < V4 * 4; ++e) x[e] = bf16_bits_to_float(float_to_bf16_bits(__fmul_rn(x[e], inv)));
}

__device__ __forceinline__ void gate_inputs(float a, float b, float A_log, float dt_bias, float &g, float &beta) {
    const float x = __fadd_rn(a, dt_bias);
    const float sp = x > 20.f ? x : log1pf(expf(x));
    g = __fmul_rn(-expf(A_log), sp);
    beta = __frcp_rn(__fadd_rn(1.f, expf(-b)));
}

// k . q over the full head dim; identical bits on all lanes of the octet.
template <int V4>
__device__ __forceinline__ float octet_dot(const float (&kk)[V4 * 4], const float (&qq)[V4 * 4]) {
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < V4 * 4; ++e) acc = fmaf(kk[e], qq[e], acc);
    return octet_sum(acc);
}

// Packed fp32x2 arithmetic (round to nearest, as two separate fp32
// operations would give): d = a * b + c and d = a * b on element pairs.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// u_j and o_j with every rounding explicit, so that the kernels sharing them
// give the same bits whatever the compiler contracts or shares around them.
__device__ __forceinline__ float row_u(float beta, float vj, float alpha, float a) {
    return __fmul_rn(beta, __fmaf_rn(-alpha, a, vj));
}
__device__ __forceinline__ float row_o(float scale, float u, float kq, float alpha, float b) {
    return __fmul_rn(scale, __fmaf_rn(u, kq, __fmul_rn(alpha, b)));
}

// Updates the lane's slice of one row in place and returns o_j.  The two dot
// products run as packed pairs: even and odd elements of the slice are summed
// in separate halves, which are added before the octet reduction.
template <int V4>
__device__ __forceinline__ float update_row(float4 (&s)[V4], const float (&kk)[V4 * 4],
                                            const float (&qq)[V4 * 4], float alpha, float beta,
                                            float vj, float kq, float scale) {
    float2 a2 = make_float2(0.f, 0.f), b2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int m = 0; m < V4; ++m) {
        const float2 s01 = make_float2(s[m].x, s[m].y), s23 = make_float2(s[m].z, s[m].w);
        a2 = fma2(s01, make_float2(kk[4 * m + 0], kk[4 * m + 1]), a2);
        b2 = fma2(s01, make_float2(qq[4 * m + 0], qq[4 * m + 1]), b2);
        a2 = fma2(s23, make_float2(kk[4 * m + 2], kk[4 * m + 3]), a2);
        b2 = fma2(s23, make_float2(qq[4 * m + 2], qq[4 * m + 3]), b2);
    }
    const float a = octet_sum(a2.x + a2.y);
    const float b = octet_sum(b2.x + b2.y);
    const float u = row_u(beta, vj, alpha, a);
    const float2 al = make_float2(alpha, alpha), uu = make_float2(u, u);
#pragma unroll
    for (int m = 0; m < V4; ++m) {
        const float2 s01 = fma2(make_float2(kk[4 * m + 0], kk[4 * m + 1]), uu, mul2(al, make_float2(s[m].x, s[m].y)));
        const float2 s23 = fma2(make_float2(kk[4 * m + 2], kk[4 * m + 3]), uu, mul2(al, make_float2(s[m].z, s[m].w)));
        s[m] = make_float4(s01.x, s01.y, s23.x, s23.y);
    }
    return row_o(scale, u, kq, alpha, b);
}

// update_row on G rows at once, phase by phase (all dot products, then the G
// pairs of octet reductions level by level, then all updates), so that the
// rows' independent dependency chains overlap.  Each row's arithmetic is
// update_row's, operation for operation: the results are the same bits.
template <int V4, int G>
__device__ __forceinline__ void update_rows(float4 (&s)[G][V4], const float (&kk)[V4 * 4],
                                            const float (&qq)[V4 * 4], float alpha, float beta,
                                            const float (&vj)[G], float kq, float scale, float (&oj)[G]) {
    float a[G], b[G];
#pragma unroll
    for (int i = 0; i < G; ++i) {
        float2 a2 = make_float2(0.f, 0.f), b2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < V4; ++m) {
            const float2 s01 = make_float2(s[i][m].x, s[i][m].y), s23 = make_float2(s[i][m].z, s[i][m].w);
            a2 = fma2(s01, make_float2(kk[4 * m + 0], kk[4 * m + 1]), a2);
            b2 = fma2(s01, make_float2(qq[4 * m + 0], qq[4 * m + 1]), b2);
            a2 = fma2(s23, make_float2(kk[4 * m + 2], kk[4 * m + 3]), a2);
            b2 = fma2(s23, make_float2(qq[4 * m + 2], qq[4 * m + 3]), b2);
        }
        a[i] = a2.x + a2.y;
        b[i] = b2.x + b2.y;
    }
#pragma unroll
    for (int lvl = 4; lvl >= 1; lvl >>= 1) {
#pragma unroll
        for (int i = 0; i < G; ++i) {
            a[i] += __shfl_xor_sync(0xffffffffu, a[i], lvl);
            b[i] += __shfl_xor_sync(0xffffffffu, b[i], lvl);
        }
    }
#pragma unroll
    for (int i = 0; i < G; ++i) {
        const float u = row_u(beta, vj[i], alpha, a[i]);
        const float2 al = make_float2(alpha, alpha), uu = make_float2(u, u);
#pragma unroll
        for (int m = 0; m < V4; ++m) {
            const float2 s01 =
                fma2(make_float2(kk[4 * m + 0], kk[4 * m + 1]), uu, mul2(al, make_float2(s[i][m].x, s[i][m].y)));
            const float2 s23 =
                fma2(make_float2(kk[4 * m + 2], kk[4 * m + 3]), uu, mul2(al, make_float2(s[i][m].z, s[i][m].w)));
            s[i][m] = make_float4(s01.x, s01.y, s23.x, s23.y);
        }
        oj[i] = row_o(scale, u, kq, alpha, b[i]);
    }
}

// update_rows for the four rows of a lane octet's 16-row item (rows
// 4 i + octet, i = 0..3) with the eight octet reductions done as one
// reduce-scatter: at each xor level (4, 2, 1) a lane keeps half of its partial
// sums and sends the other half to its partner, so that lane l8 ends with
// a_{l8} (l8 < 4) or b_{l8-4} (l8 >= 4).  Each sum is built from the same
// pairs in the same order as octet_sum's butterfly, so it has the same bits.
// u_i is formed on lane i of the octet and broadcast; o of row l8 & 3 is
// returned on lanes l8 >= 4.  vj_own is v of row l8 & 3.
template <int V4>
__device__ __forceinline__ float update_rows4_scatter(float4 (&s)[4][V4], const float (&kk)[V4 * 4],
                                                      const float (&qq)[V4 * 4], float alpha, float beta,
                                                      float vj_own, float kq, float scale, int lane) {
    const int l8 = lane & 7, base = lane & ~7;
    float a[4], b[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 a2 = make_float2(0.f, 0.f), b2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < V4; ++m) {
            const float2 s01 = make_float2(s[i][m].x, s[i][m].y), s23 = make_float2(s[i][m].z, s[i][m].w);
            a2 = fma2(s01, make_float2(kk[4 * m + 0], kk[4 * m + 1]), a2);
            b2 = fma2(s01, make_float2(qq[4 * m + 0], qq[4 * m + 1]), b2);
            a2 = fma2(s23, make_float2(kk[4 * m + 2], kk[4 * m + 3]), a2);
            b2 = fma2(s23, make_float2(qq[4 * m + 2], qq[4 * m + 3]), b2);
        }
        a[i] = a2.x + a2.y;
        b[i] = b2.x + b2.y;
    }
    const bool h4 = l8 & 4, h2 = l8 & 2, h1 = l8 & 1;
    float c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = h4 ? a[i] : b[i];
        c[i] = (h4 ? b[i] : a[i]) + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    float d[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = h2 ? c[i] : c[i + 2];
        d[i] = (h2 ? c[i + 2] : c[i]) + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    const float e = (h1 ? d[1] : d[0]) + __shfl_xor_sync(0xffffffffu, h1 ? d[0] : d[1], 1);
    const float u_own = row_u(beta, vj_own, alpha, e);  // meaningful on lanes l8 < 4
    float u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) u[i] = __shfl_sync(0xffffffffu, u_own, base | i);
    const float u_row = __shfl_sync(0xffffffffu, u_own, base | (l8 & 3));
    const float o = row_o(scale, u_row, kq, alpha, e);  // meaningful on lanes l8 >= 4
    const float2 al = make_float2(alpha, alpha);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 uu = make_float2(u[i], u[i]);
#pragma unroll
        for (int m = 0; m < V4; ++m) {
            const float2 s01 =
                fma2(make_float2(kk[4 * m + 0], kk[4 * m + 1]), uu, mul2(al, make_float2(s[i][m].x, s[i][m].y)));
            const float2 s23 =
                fma2(make_float2(kk[4 * m + 2], kk[4 * m + 3]), uu, mul2(al, make_float2(s[i][m].z, s[i][m].w)));
            s[i][m] = make_float4(s01.x, s01.y, s23.x, s23.y);
        }
    }
    return o;
}

}  // namespace gdn
