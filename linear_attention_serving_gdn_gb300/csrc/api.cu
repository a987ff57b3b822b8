// C ABI of libgdn: host-side validation, then kernel launches on the caller's
// stream.  See include/gdn.h for the contract of each entry point.
#include <limits.h>

#include "gdn_internal.cuh"

namespace gdn {

bool current_device(int *dev, int *sms) {
    static int cache[kMaxDevices] = {};
    if (cudaGetDevice(dev) != cudaSuccess) return false;
    if (*dev >= 0 && *dev < kMaxDevices && __atomic_load_n(&cache[*dev], __ATOMIC_ACQUIRE) > 0) {
        *sms = cache[*dev];
        return true;
    }
    if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess || *sms < 1)
        return false;
    if (*dev >= 0 && *dev < kMaxDevices) __atomic_store_n(&cache[*dev], *sms, __ATOMIC_RELEASE);
    return true;
}

}  // namespace gdn

namespace {

using gdn::kChunk;

bool dims_ok(const gdn_dims_t *d, gdn_status_t *why) {
    if (!d) {
        *why = GDN_ERR_INVALID_ARG;
        return false;
    }
    if (d->h_k <= 0 || d->h_v <= 0 || d->d_k <= 0 || d->d_v <= 0 || d->h_v % d->h_k != 0) {
        *why = GDN_ERR_INVALID_ARG;
        return false;
    }
    if (d->d_k != d->d_v || (d->d_k != 64 && d->d_k != 128)) {
        *why = GDN_ERR_UNSUPPORTED;
        return false;
    }
    return true;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Validates a host cu_seqlens mirror: starts at 0, non-decreasing.
bool cu_ok(const int32_t *cu, int32_t n) {
    if (!cu || cu[0] != 0) return false;
    for (int32_t i = 0; i < n; ++i)
        if (cu[i + 1] < cu[i]) return false;
    return true;
}

int64_t num_emits(const int32_t *cu, int32_t n, int32_t E) {
    if (E <= 0) return 0;
    int64_t tot = 0;
    for (int32_t i = 0; i < n; ++i) tot += (cu[i + 1] - cu[i]) / (static_cast<int64_t>(kChunk) * E);
    return tot;
}

// Raw-input preparation parameters of the fused decode (all null: none).
struct RawPrep {
    const float *a = nullptr, *b = nullptr, *A_log = nullptr, *dt_bias = nullptr;
    float eps = 0.f;
};

// Validates a decode call and fills its kernel arguments; launches nothing.
gdn_status_t decode_check(const gdn_dims_t *dims, int32_t num_rows, const gdn_bf16 *q,
                          const gdn_bf16 *k, const gdn_bf16 *v, const float *g, const float *beta,
                          float *state, int64_t num_slots, const int32_t *src_slot,
                          const int32_t *dst_slot, gdn_bf16 *o, int32_t *dev_status,
                          gdn::DecodeArgs *out, const RawPrep &raw = RawPrep()) {
    gdn_status_t why = GDN_OK;
    if (!dims_ok(dims, &why)) return why;
    if (num_rows < 0 || num_slots < 0) return GDN_ERR_INVALID_ARG;
    if (num_rows == 0) return GDN_OK;
    const bool have_gates = raw.a ? (raw.b && raw.A_log && raw.dt_bias && raw.eps >= 0.f) : (g && beta);
    if (!q || !k || !v || !have_gates || !state || !src_slot || !o) return GDN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(state) || !aligned16(o))
        return GDN_ERR_INVALID_ARG;
    gdn::DecodeArgs &a = *out;
    a.num_rows = num_rows;
    a.h_k = dims->h_k;
    a.h_v = dims->h_v;
    a.scale = dims->scale;
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = g;
    a.beta = beta;
    a.state = state;
    a.num_slots = num_slots;
    a.src_slot = src_slot;
    a.dst_slot = dst_slot;
    a.o = o;
    a.dev_status = dev_status;
    a.a_raw = raw.a;
    a.b_raw = raw.b;
    a.A_log = raw.A_log;
    a.dt_bias = raw.dt_bias;
    a.eps = raw.eps;
    return GDN_OK;
}

gdn_status_t decode_impl(const gdn_dims_t *dims, int32_t num_rows, const gdn_bf16 *q,
                         const gdn_bf16 *k, const gdn_bf16 *v, const float *g, const float *beta,
                         float *state, int64_t num_slots, const int32_t *src_slot,
                         const int32_t *dst_slot, gdn_bf16 *o, int32_t *dev_status,
                         cudaStream_t stream, const RawPrep &raw = RawPrep()) {
    gdn::DecodeArgs a{};
    const gdn_status_t s = decode_check(dims, num_rows, q, k, v, g, beta, state, num_slots, src_slot,
                                        dst_slot, o, dev_status, &a, raw);
    if (s != GDN_OK || num_rows == 0) return s;
    return gdn::launch_decode(a, dims->d_k, stream) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status_t decode_multi_impl(const gdn_dims_t *dims, int32_t num_rows, int32_t tokens_per_row,
                               const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                               const float *g, const float *beta, float *state, int64_t num_slots,
                               const int32_t *src_slot, const int32_t *dst_slots, gdn_bf16 *o,
                               int32_t *dev_status, cudaStream_t stream) {
    gdn_status_t why = GDN_OK;
    if (!dims_ok(dims, &why)) return why;
    if (num_rows < 0 || tokens_per_row < 1 || num_slots < 0) return GDN_ERR_INVALID_ARG;
    if (static_cast<int64_t>(num_rows) * tokens_per_row > INT_MAX) return GDN_ERR_UNSUPPORTED;
    if (num_rows == 0) return GDN_OK;
    if (!q || !k || !v || !g || !beta || !state || !src_slot || !o) return GDN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(state) || !aligned16(o))
        return GDN_ERR_INVALID_ARG;
    gdn::DecodeMultiArgs a;
    a.num_rows = num_rows;
    a.tokens_per_row = tokens_per_row;
    a.h_k = dims->h_k;
    a.h_v = dims->h_v;
    a.scale = dims->scale;
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = g;
    a.beta = beta;
    a.state = state;
    a.num_slots = num_slots;
    a.src_slot = src_slot;
    a.dst_slots = dst_slots;
    a.o = o;
    a.dev_status = dev_status;
    return gdn::launch_decode_multi(a, dims->d_k, stream) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// Largest emission stride: 64 E stays far inside int32 on the device.
constexpr int32_t kMaxEmitEvery = 1 << 24;

size_t workspace_need(const gdn_dims_t *, int32_t, int64_t) { return 0; }

gdn_status_t workspace_ok(const gdn_dims_t *dims, int32_t num_seqs, int64_t T, const void *ws,
                          size_t ws_bytes) {
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return GDN_ERR_WORKSPACE;
    const size_t need = workspace_need(dims, num_seqs, T);
    if (need > 0 && (!ws || ws_bytes < need)) return GDN_ERR_WORKSPACE;
    return GDN_OK;
}

// Validates a prefill call and fills its kernel arguments; launches nothing.
gdn_status_t prefill_check(const gdn_dims_t *dims, int32_t num_seqs, const int32_t *cu_seqlens,
                           const int32_t *cu_host, const gdn_bf16 *q, const gdn_bf16 *k,
                           const gdn_bf16 *v, const float *g, const float *beta, float *state,
                           int64_t num_slots, const int32_t *src_slot, const int32_t *dst_slot,
                           gdn_bf16 *o, float *chunk_states, int32_t E, int64_t capacity,
                           const void *workspace, size_t workspace_bytes, int32_t *dev_status,
                           gdn::PrefillArgs *out, const int32_t *emit_table = nullptr,
                           int32_t emit_table_stride = 0, const int32_t *emit_first = nullptr) {
    gdn_status_t why = GDN_OK;
    if (!dims_ok(dims, &why)) return why;
    if (num_seqs < 0 || num_slots < 0 || E < 0 || E > kMaxEmitEvery) return GDN_ERR_INVALID_ARG;
    if (emit_table && (!emit_first || emit_table_stride < 1 || !state)) return GDN_ERR_INVALID_ARG;
    if (num_seqs == 0) return GDN_OK;
    if (!cu_seqlens || !cu_ok(cu_host, num_seqs)) return GDN_ERR_INVALID_ARG;
    const int64_t T = cu_host[num_seqs];
    if ((src_slot || dst_slot) && !state) return GDN_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !g || !beta || !o)) return GDN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(state) || !aligned16(o) ||
        !aligned16(chunk_states))
        return GDN_ERR_INVALID_ARG;
    if (E > 0 && !emit_table) {
        const int64_t need = num_emits(cu_host, num_seqs, E);
        if (need > 0 && (!chunk_states || capacity < need)) return GDN_ERR_INVALID_ARG;
    }
    if (static_cast<int64_t>(num_seqs) * dims->h_v > INT_MAX) return GDN_ERR_UNSUPPORTED;
    const gdn_status_t ws = workspace_ok(dims, num_seqs, T, workspace, workspace_bytes);
    if (ws != GDN_OK) return ws;
    gdn::PrefillArgs &a = *out;
    a.num_seqs = num_seqs;
    a.h_k = dims->h_k;
    a.h_v = dims->h_v;
    a.scale = dims->scale;
    a.cu_seqlens = cu_seqlens;
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = g;
    a.beta = beta;
    a.state = state;
    a.num_slots = num_slots;
    a.src_slot = src_slot;
    a.dst_slot = dst_slot;
    a.o = o;
    a.chunk_states = (E > 0 && !emit_table) ? chunk_states : nullptr;
    a.emit_every_chunks = E;
    a.dev_status = dev_status;
    a.total_tokens = T;
    a.chunk_capacity = (E > 0 && !emit_table) ? capacity : 0;
    a.emit_table = E > 0 ? emit_table : nullptr;
    a.emit_first = E > 0 ? emit_first : nullptr;
    a.emit_table_stride = emit_table_stride;
    return GDN_OK;
}

gdn_status_t prefill_impl(const gdn_dims_t *dims, int32_t num_seqs, const int32_t *cu_seqlens,
                          const int32_t *cu_host, const gdn_bf16 *q, const gdn_bf16 *k,
                          const gdn_bf16 *v, const float *g, const float *beta, float *state,
                          int64_t num_slots, const int32_t *src_slot, const int32_t *dst_slot,
                          gdn_bf16 *o, float *chunk_states, int32_t E, int64_t capacity,
                          const void *workspace, size_t workspace_bytes, int32_t *dev_status,
                          cudaStream_t stream, const int32_t *emit_table = nullptr,
                          int32_t emit_table_stride = 0, const int32_t *emit_first = nullptr) {
    gdn::PrefillArgs a{};
    const gdn_status_t s = prefill_check(dims, num_seqs, cu_seqlens, cu_host, q, k, v, g, beta, state,
                                         num_slots, src_slot, dst_slot, o, chunk_states, E, capacity,
                                         workspace, workspace_bytes, dev_status, &a, emit_table,
                                         emit_table_stride, emit_first);
    if (s != GDN_OK || num_seqs == 0) return s;
    return gdn::launch_prefill(a, dims->d_k, cu_host, stream) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

extern "C" {

gdn_status_t gdn_decode_packed(const gdn_dims_t *dims, int32_t num_rows, const gdn_bf16 *q,
                               const gdn_bf16 *k, const gdn_bf16 *v, const float *g,
                               const float *beta, float *state, int64_t num_slots,
                               const int32_t *src_slot, const int32_t *dst_slot, gdn_bf16 *o,
                               int32_t *dev_status, void *stream) {
    return decode_impl(dims, num_rows, q, k, v, g, beta, state, num_slots, src_slot, dst_slot, o,
                       dev_status, static_cast<cudaStream_t>(stream));
}

gdn_status_t gdn_decode_packed_raw(const gdn_dims_t *dims, int32_t num_rows, const gdn_bf16 *q_raw,
                                   const gdn_bf16 *k_raw, const gdn_bf16 *v, const float *a,
                                   const float *b, const float *A_log, const float *dt_bias, float eps,
                                   float *state, int64_t num_slots, const int32_t *src_slot,
                                   const int32_t *dst_slot, gdn_bf16 *o, int32_t *dev_status,
                                   void *stream) {
    if (!a || !b || !A_log || !dt_bias || !(eps >= 0.f)) return GDN_ERR_INVALID_ARG;
    RawPrep raw;
    raw.a = a;
    raw.b = b;
    raw.A_log = A_log;
    raw.dt_bias = dt_bias;
    raw.eps = eps;
    return decode_impl(dims, num_rows, q_raw, k_raw, v, nullptr, nullptr, state, num_slots, src_slot,
                       dst_slot, o, dev_status, static_cast<cudaStream_t>(stream), raw);
}

gdn_status_t gdn_prep_inputs(const gdn_dims_t *dims, int64_t num_tokens, const gdn_bf16 *q_raw,
                             const gdn_bf16 *k_raw, const float *a, const float *b, const float *A_log,
                             const float *dt_bias, float eps, gdn_bf16 *q, gdn_bf16 *k, float *g,
                             float *beta, void *stream) {
    gdn_status_t why = GDN_OK;
    if (!dims_ok(dims, &why)) return why;
    if (num_tokens < 0 || !(eps >= 0.f)) return GDN_ERR_INVALID_ARG;
    if (num_tokens == 0) return GDN_OK;
    if (!q_raw || !k_raw || !a || !b || !A_log || !dt_bias || !q || !k || !g || !beta) return GDN_ERR_INVALID_ARG;
    if (!aligned16(q_raw) || !aligned16(k_raw) || !aligned16(q) || !aligned16(k)) return GDN_ERR_INVALID_ARG;
    gdn::PrepArgs p;
    p.num_tokens = num_tokens;
    p.h_k = dims->h_k;
    p.h_v = dims->h_v;
    p.q_raw = q_raw;
    p.k_raw = k_raw;
    p.a = a;
    p.b = b;
    p.A_log = A_log;
    p.dt_bias = dt_bias;
    p.eps = eps;
    p.q = q;
    p.k = k;
    p.g = g;
    p.beta = beta;
    return gdn::launch_prep(p, dims->d_k, static_cast<cudaStream_t>(stream)) == cudaSuccess ? GDN_OK
                                                                                             : GDN_ERR_CUDA;
}

gdn_status_t gdn_decode_multi(const gdn_dims_t *dims, int32_t num_rows, int32_t tokens_per_row,
                              const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                              const float *g, const float *beta, float *state, int64_t num_slots,
                              const int32_t *src_slot, const int32_t *dst_slots, gdn_bf16 *o,
                              int32_t *dev_status, void *stream) {
    return decode_multi_impl(dims, num_rows, tokens_per_row, q, k, v, g, beta, state, num_slots,
                             src_slot, dst_slots, o, dev_status, static_cast<cudaStream_t>(stream));
}

gdn_status_t gdn_prefill_varlen(const gdn_dims_t *dims, int32_t num_seqs,
                                const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                                const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                                const float *g, const float *beta, float *state,
                                int64_t num_slots, const int32_t *src_slot,
                                const int32_t *dst_slot, gdn_bf16 *o, float *chunk_states,
                                int32_t emit_every_chunks, int64_t chunk_states_capacity,
                                void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                void *stream) {
    return prefill_impl(dims, num_seqs, cu_seqlens, cu_seqlens_host, q, k, v, g, beta, state,
                        num_slots, src_slot, dst_slot, o, chunk_states, emit_every_chunks,
                        chunk_states_capacity, workspace, workspace_bytes, dev_status,
                        static_cast<cudaStream_t>(stream));
}

size_t gdn_prefill_workspace_bytes(const gdn_dims_t *dims, int32_t num_seqs, int64_t total_tokens) {
    gdn_status_t why = GDN_OK;
    if (!dims_ok(dims, &why) || num_seqs < 0 || total_tokens < 0) return static_cast<size_t>(-1);
    return workspace_need(dims, num_seqs, total_tokens);
}

gdn_status_t gdn_prefill_varlen_apc(const gdn_dims_t *dims, int32_t num_seqs,
                                    const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                                    const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                                    const float *g, const float *beta, float *state,
                                    int64_t num_slots, const int32_t *src_slot,
                                    const int32_t *dst_slot, gdn_bf16 *o,
                                    int32_t emit_every_chunks, const int32_t *block_table,
                                    int32_t block_table_stride, const int32_t *block_first,
                                    void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                    void *stream) {
    if (emit_every_chunks < 1 || !block_table || !block_first || block_table_stride < 1 || !state)
        return GDN_ERR_INVALID_ARG;
    return prefill_impl(dims, num_seqs, cu_seqlens, cu_seqlens_host, q, k, v, g, beta, state,
                        num_slots, src_slot, dst_slot, o, nullptr, emit_every_chunks, 0, workspace,
                        workspace_bytes, dev_status, static_cast<cudaStream_t>(stream), block_table,
                        block_table_stride, block_first);
}

namespace {

// Both halves of a mixed step validated, then launched: the decode rows on
// `dec_st` and the prefill on `st`; with a separate `dec_st`, the two are
// forked from and joined back into `st` through the caller's events.
gdn_status_t mixed_impl(const gdn_dims_t *dims, int32_t num_decodes, int32_t num_prefills,
                        const int32_t *cu_seqlens_p, const int32_t *cu_seqlens_p_host,
                        const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                        const float *g, const float *beta, float *state, int64_t num_slots,
                        const int32_t *dec_src_slot, const int32_t *dec_dst_slot,
                        const int32_t *pre_src_slot, const int32_t *pre_dst_slot,
                        gdn_bf16 *o, float *chunk_states, int32_t emit_every_chunks,
                        int64_t chunk_states_capacity, void *workspace, size_t workspace_bytes,
                        int32_t *dev_status, cudaStream_t st, cudaStream_t dec_st,
                        cudaEvent_t fork_event, cudaEvent_t join_event) {
    gdn_status_t why = GDN_OK;
    if (!dims_ok(dims, &why)) return why;
    if (num_decodes < 0 || num_prefills < 0) return GDN_ERR_INVALID_ARG;
    if (num_prefills > 0 && !cu_ok(cu_seqlens_p_host, num_prefills)) return GDN_ERR_INVALID_ARG;
    if (num_decodes > 0 && (!dec_src_slot || !state)) return GDN_ERR_INVALID_ARG;
    if (num_prefills > 0 && !cu_seqlens_p) return GDN_ERR_INVALID_ARG;
    const bool forked = dec_st != st;
    if (forked && (!fork_event || !join_event)) return GDN_ERR_INVALID_ARG;
    // The prefill part starts num_decodes rows into every token-major tensor;
    // rows are 16-byte multiples for the supported head dims.
    const size_t hk = static_cast<size_t>(dims->h_k) * dims->d_k;
    const size_t hv = static_cast<size_t>(dims->h_v) * dims->d_v;
    const size_t nd = static_cast<size_t>(num_decodes);
    auto off16 = [&](const gdn_bf16 *p, size_t row) { return p ? p + nd * row : nullptr; };
    auto offf = [&](const float *p) { return p ? p + nd * dims->h_v : nullptr; };
    // Both halves are validated completely before either is launched.
    gdn::DecodeArgs da{};
    gdn_status_t s = decode_check(dims, num_decodes, q, k, v, g, beta, state, num_slots, dec_src_slot,
                                  dec_dst_slot, o, dev_status, &da);
    if (s != GDN_OK) return s;
    gdn::PrefillArgs pa{};
    s = prefill_check(dims, num_prefills, cu_seqlens_p, cu_seqlens_p_host, off16(q, hk), off16(k, hk),
                      off16(v, hv), offf(g), offf(beta), state, num_slots, pre_src_slot, pre_dst_slot,
                      o ? o + nd * hv : nullptr, chunk_states, emit_every_chunks, chunk_states_capacity,
                      workspace, workspace_bytes, dev_status, &pa);
    if (s != GDN_OK) return s;
    if (forked && (cudaEventRecord(fork_event, st) != cudaSuccess ||
                   cudaStreamWaitEvent(dec_st, fork_event, 0) != cudaSuccess))
        return GDN_ERR_CUDA;
    if (num_decodes > 0 && gdn::launch_decode(da, dims->d_k, dec_st) != cudaSuccess) return GDN_ERR_CUDA;
    if (num_prefills > 0 && gdn::launch_prefill(pa, dims->d_k, cu_seqlens_p_host, st) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (forked && (cudaEventRecord(join_event, dec_st) != cudaSuccess ||
                   cudaStreamWaitEvent(st, join_event, 0) != cudaSuccess))
        return GDN_ERR_CUDA;
    return GDN_OK;
}

}  // namespace

gdn_status_t gdn_mixed_step(const gdn_dims_t *dims, int32_t num_decodes, int32_t num_prefills,
                            const int32_t *cu_seqlens_p, const int32_t *cu_seqlens_p_host,
                            const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                            const float *g, const float *beta, float *state, int64_t num_slots,
                            const int32_t *dec_src_slot, const int32_t *dec_dst_slot,
                            const int32_t *pre_src_slot, const int32_t *pre_dst_slot,
                            gdn_bf16 *o, float *chunk_states, int32_t emit_every_chunks,
                            int64_t chunk_states_capacity, void *workspace, size_t workspace_bytes,
                            int32_t *dev_status, void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return mixed_impl(dims, num_decodes, num_prefills, cu_seqlens_p, cu_seqlens_p_host, q, k, v, g, beta, state,
                      num_slots, dec_src_slot, dec_dst_slot, pre_src_slot, pre_dst_slot, o, chunk_states,
                      emit_every_chunks, chunk_states_capacity, workspace, workspace_bytes, dev_status, st, st,
                      nullptr, nullptr);
}

gdn_status_t gdn_mixed_step_colaunch(const gdn_dims_t *dims, int32_t num_decodes, int32_t num_prefills,
                                     const int32_t *cu_seqlens_p, const int32_t *cu_seqlens_p_host,
                                     const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                                     const float *g, const float *beta, float *state, int64_t num_slots,
                                     const int32_t *dec_src_slot, const int32_t *dec_dst_slot,
                                     const int32_t *pre_src_slot, const int32_t *pre_dst_slot,
                                     gdn_bf16 *o, float *chunk_states, int32_t emit_every_chunks,
                                     int64_t chunk_states_capacity, void *workspace, size_t workspace_bytes,
                                     int32_t *dev_status, void *stream, void *aux_stream, void *fork_event,
                                     void *join_event) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaStream_t dec_st = aux_stream ? static_cast<cudaStream_t>(aux_stream) : st;
    return mixed_impl(dims, num_decodes, num_prefills, cu_seqlens_p, cu_seqlens_p_host, q, k, v, g, beta, state,
                      num_slots, dec_src_slot, dec_dst_slot, pre_src_slot, pre_dst_slot, o, chunk_states,
                      emit_every_chunks, chunk_states_capacity, workspace, workspace_bytes, dev_status, st, dec_st,
                      static_cast<cudaEvent_t>(fork_event), static_cast<cudaEvent_t>(join_event));
}

int64_t gdn_prefill_num_emits(const int32_t *cu_seqlens_host, int32_t num_seqs,
                              int32_t emit_every_chunks) {
    if (num_seqs < 0 || (num_seqs > 0 && !cu_ok(cu_seqlens_host, num_seqs))) return -1;
    return num_emits(cu_seqlens_host, num_seqs, emit_every_chunks);
}

gdn_status_t gdn_prefill_emit_offsets(const int32_t *cu_seqlens_host, int32_t num_seqs,
                                      int32_t emit_every_chunks, int64_t *out) {
    if (!out || num_seqs < 0 || (num_seqs > 0 && !cu_ok(cu_seqlens_host, num_seqs)))
        return GDN_ERR_INVALID_ARG;
    out[0] = 0;
    for (int32_t i = 0; i < num_seqs; ++i)
        out[i + 1] = out[i] + (emit_every_chunks > 0
                                   ? (cu_seqlens_host[i + 1] - cu_seqlens_host[i]) /
                                         (static_cast<int64_t>(kChunk) * emit_every_chunks)
                                   : 0);
    return GDN_OK;
}

int32_t gdn_align_block_size(int32_t block_size) {
    if (block_size <= 0 || block_size > INT_MAX - kChunk) return -1;
    return (block_size + kChunk - 1) / kChunk * kChunk;
}

int32_t gdn_grid_emit_every_chunks(int32_t block_size) {
    const int32_t b = gdn_align_block_size(block_size);
    return b < 0 ? -1 : b / kChunk;  // lcm(64, b) == b once b is a multiple of 64
}

int64_t gdn_floor_prefix_hit(int64_t hit_tokens, int64_t prompt_tokens, int32_t block_size) {
    const int32_t b = gdn_align_block_size(block_size);
    if (b < 0 || hit_tokens < 0 || prompt_tokens < 0 || hit_tokens > prompt_tokens) return -1;
    if (hit_tokens == prompt_tokens) return hit_tokens;
    return hit_tokens / b * b;
}

gdn_status_t gdn_status_from_device(int32_t word) {
    if (word & GDN_DEV_TIMEOUT) return GDN_ERR_TIMEOUT;
    if (word != 0) return GDN_ERR_INVALID_ARG;
    return GDN_OK;
}

const char *gdn_status_string(gdn_status_t status) {
    switch (status) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG: invalid argument";
        case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: unsupported shape";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA: CUDA launch or runtime error";
        case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE: workspace too small or misaligned";
        case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT: a bounded device wait expired";
    }
    return "unknown gdn_status_t";
}

}  // extern "C"
