// C ABI of libgdn.so (declared in include/gdn.h): argument validation, launch
// planning and status codes.  Every check runs before the first enqueue, so a
// rejected call enqueues nothing; nothing here allocates or synchronises.
#include <atomic>
#include <climits>
#include <cstdint>
#include <cstring>

#include "gdn_common.cuh"
#include "rows_common.cuh"
#include "gdn_tc.cuh"

namespace {

thread_local int g_last_cuda_error = 0;

bool head_dim_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return GDN_OK;
    g_last_cuda_error = int(e);
    return GDN_ERR_CUDA;
}

size_t elem_size(int dtype) { return dtype == GDN_FP32 ? 4 : 2; }

int64_t conv_channels(const gdn_prefill_desc* d) {
    return 2 * int64_t(d->Hk) * d->dk + int64_t(d->Hv) * d->dv;
}

// Shape, dtype and option checks shared by prefill and step.
int check_common(const gdn_prefill_desc* d) {
    if (d == nullptr) return GDN_ERR_INVALID_ARG;
    if (d->dtype != GDN_BF16 && d->dtype != GDN_FP32) return GDN_ERR_UNSUPPORTED;
    if (d->B < 0 || d->Hk <= 0 || d->Hv <= 0) return GDN_ERR_INVALID_ARG;
    if (d->Hv % d->Hk != 0) return GDN_ERR_UNSUPPORTED;
    if (!head_dim_ok(d->dk) || !head_dim_ok(d->dv)) return GDN_ERR_UNSUPPORTED;
    if (d->B > 65535 || d->Hv > 65535) return GDN_ERR_TOO_LARGE;
    if (d->use_qk_l2norm && !(d->l2_eps >= 0.f)) return GDN_ERR_INVALID_ARG;
    if (d->conv_x != nullptr) {
        if (d->conv_w == nullptr) return GDN_ERR_INVALID_ARG;
        if (d->conv_kernel < 2 || d->conv_kernel > 8) return GDN_ERR_UNSUPPORTED;
        if (d->conv_act != GDN_ACT_NONE && d->conv_act != GDN_ACT_SILU) return GDN_ERR_UNSUPPORTED;
        if (!aligned16(d->conv_x)) return GDN_ERR_ALIGN;
    }
    if (d->g == nullptr || d->beta == nullptr || d->out == nullptr) return GDN_ERR_INVALID_ARG;
    if (d->conv_x == nullptr && (d->q == nullptr || d->k == nullptr || d->v == nullptr))
        return GDN_ERR_INVALID_ARG;
    if (d->conv_x == nullptr && (!aligned16(d->q) || !aligned16(d->k) || !aligned16(d->v)))
        return GDN_ERR_ALIGN;
    if (!aligned16(d->out) || !aligned16(d->state_in) || !aligned16(d->state_out))
        return GDN_ERR_ALIGN;
    return GDN_OK;
}

size_t conv_workspace(const gdn_prefill_desc* d) {
    if (d->conv_x == nullptr || d->T_total <= 0) return 0;
    const size_t bytes = size_t(d->T_total) * size_t(conv_channels(d)) * elem_size(d->dtype);
    return (bytes + 255) & ~size_t(255);
}

// Streaming multiprocessors of the current device (cudaDevAttrMultiProcessorCount,
// looked up once per device); 152, a GB300's count, where no device answers
// (host-only planning, as in gdn_workspace_bytes on a machine without a GPU).
int sm_count() {
    constexpr int kFallback = 152;
    constexpr int kMaxDevices = 64;
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return kFallback;
    }
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return kFallback;
    }
    cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

// seg_out_kernel's work per (sequence, value head), in chunk periods of the
// state pass: a CTA of segment s takes s - 1 state steps (kSoStep each) and
// then its chunk group's outputs (kSoOut each).
constexpr double kSoStep = 1.0, kSoOut = 0.35;

// seg_out_kernel's CTAs per (sequence, value head): one per chunk group of
// every segment s >= 1, plus one for the final state, as many as fit one
// wave.  Each segment starts with one group; the remaining CTAs go one by one
// to the segment whose CTAs finish last (the later a segment, the more state
// steps precede its outputs), at most one group per chunk.  When even one
// group per segment leaves no room for the final state's CTA, the last
// group's CTA of the last segment forms it after its outputs
// (*final_cta = 0).  gstart (seg_max entries, may be null) receives the
// first CTA of every segment s >= 1 (gstart[s - 1]) and their total
// (gstart[seg_max - 1]); *groups the uniform group count used beyond the
// table.  Returns the cost of the slowest CTA.
double seg_out_plan(int64_t units, int64_t seg_max, int seg_chunks, int* final_cta, int* groups,
                    int16_t* gstart) {
    *final_cta = 1;
    *groups = 1;
    if (seg_max < 2) return 0.0;
    const int64_t per_unit = sm_count() / units;   // CTAs per (sequence, value head) in one wave
    const int64_t nout = seg_max - 1;               // output segments
    int64_t budget;
    if (per_unit >= nout + 1) {
        budget = per_unit - 1;
    } else {
        *final_cta = 0;
        budget = per_unit > nout ? per_unit : nout;
    }
    int64_t g = budget / nout;
    if (g < 1) g = 1;
    if (g > seg_chunks) g = seg_chunks;
    *groups = int(g);
    auto cost = [&](int64_t s, int64_t gs) {
        double c = double(s - 1) * kSoStep + double((seg_chunks + gs - 1) / gs) * kSoOut;
        if (!*final_cta && s == nout) c += kSoStep;   // the final state after the outputs
        return c;
    };
    const double final_cost = *final_cta ? double(nout) * kSoStep : 0.0;
    if (nout > gdn::kSegTable) {
        const double worst = cost(nout, g);
        return worst > final_cost ? worst : final_cost;
    }
    int64_t gs[gdn::kSegTable + 1];
    for (int64_t s = 1; s <= nout; ++s) gs[s] = 1;
    for (int64_t left = budget - nout; left > 0; --left) {
        int64_t worst = 1;
        for (int64_t s = 2; s <= nout; ++s)
            if (cost(s, gs[s]) >= cost(worst, gs[worst])) worst = s;
        if (gs[worst] >= seg_chunks) break;       // its chunks cannot be split further
        ++gs[worst];
    }
    double worst = final_cost;
    int64_t z = 0;
    for (int64_t s = 1; s <= nout; ++s) {
        if (gstart) gstart[s - 1] = int16_t(z);
        z += gs[s];
        const double c = cost(s, gs[s]);
        if (c > worst) worst = c;
    }
    if (gstart) gstart[nout] = int16_t(z);
    return worst;
}

// Chunks per segment of the segment-parallel scan, or 0 for one pass.
// Cost model in chunk periods of one CTA (one CTA per SM): with n segments of
// L = ceil(chunks / n) chunks, phase 1 runs (2n - 1) CTAs per (sequence,
// value head), each taking L + kStartPeriods periods per wave of one CTA per SM
// (a CTA's first chunks run with cold instruction caches and its incoming
// state still on the way); seg_out_kernel then takes its slowest CTA's state
// steps and output chunks (seg_out_plan) per wave of its CTAs.  One pass
// costs chunks + kStartPeriods periods in ceil(units / SMs) waves.  The
// cheapest n wins; sequence lengths are taken as the batch average.
int segment_chunks(const gdn_prefill_desc* d) {
    if (d->dtype != GDN_BF16 || d->dk != 128 || d->dv != 128) return 0;   // tensor-core path only
    if (d->T_total <= 0 || d->B <= 0 || d->segment_chunks < 0) return 0;
    const int64_t chunks = (d->T_total + d->chunk - 1) / d->chunk;
    if (d->segment_chunks > 0) return d->segment_chunks < chunks ? d->segment_chunks : 0;
    constexpr double kStartPeriods = 3.0;
    const int64_t units = int64_t(d->Hv) * d->B;
    const int64_t per_seq = (chunks + d->B - 1) / d->B;
    const int64_t sms = sm_count();
    auto waves = [&](int64_t ctas) { return (ctas + sms - 1) / sms; };
    double best = double(waves(units)) * (double(per_seq) + kStartPeriods);
    int best_len = 0;
    for (int64_t n = 2; n <= 64 && n <= per_seq; ++n) {
        const int64_t len = (per_seq + n - 1) / n;
        int final_cta = 1, groups = 1;
        int16_t gstart[gdn::kSegTable + 1];
        const double worst = seg_out_plan(units, n, int(len), &final_cta, &groups, gstart);
        const int64_t so_ctas = n - 1 <= gdn::kSegTable ? gstart[n - 1] : (n - 1) * groups;
        const double out = double(waves(units * (so_ctas + final_cta))) * worst;
        const double cost = double(waves(units * (2 * n - 1))) * (double(len) + kStartPeriods) + out;
        if (cost < best) {
            best = cost;
            best_len = int(len);
        }
    }
    return best_len;
}

int64_t segment_slots(const gdn_prefill_desc* d, int seg_chunks) {
    const int64_t seg_tokens = int64_t(seg_chunks) * d->chunk;
    return d->T_total / seg_tokens + d->B + 1;
}

// The segment maps (B_s, M_s, S_s per value head and slot), then the output
// map G (bf16, one row of Hv * dv per token).
size_t segment_map_bytes(const gdn_prefill_desc* d, int seg_chunks) {
    const size_t bytes = size_t(d->Hv) * size_t(segment_slots(d, seg_chunks)) * 3 * size_t(d->dk) *
                         size_t(d->dv) * sizeof(float);
    return (bytes + 255) & ~size_t(255);
}

size_t segment_workspace(const gdn_prefill_desc* d, int seg_chunks) {
    if (seg_chunks <= 0) return 0;
    const size_t g_bytes = size_t(d->T_total) * size_t(d->Hv) * size_t(d->dv) * 2;
    return segment_map_bytes(d, seg_chunks) + ((g_bytes + 255) & ~size_t(255));
}

// Chunk records of the split preparation: one per (value head, chunk slot),
// slots t0_n / chunk + n + c (at most T_total / chunk + B + 1 per head).
int64_t prep_slots(const gdn_prefill_desc* d) { return d->T_total / d->chunk + d->B + 1; }

size_t prep_workspace(const gdn_prefill_desc* d) {
    if (d->dtype != GDN_BF16 || d->dk != 128 || d->dv != 128) return 0;   // tensor-core path only
    if (d->T_total <= 0 || d->B <= 0 || d->split_prep < 0) return 0;
    // the preparation counts its items (Hv x slots) in 32 bits
    if (int64_t(d->Hv) * prep_slots(d) >= (int64_t(1) << 31)) return 0;
    return size_t(d->Hv) * size_t(prep_slots(d)) * gdn::kPrepRecordBytes;
}

size_t workspace_needed(const gdn_prefill_desc* d) {
    return conv_workspace(d) + segment_workspace(d, segment_chunks(d)) + prep_workspace(d);
}

int check_prefill(const gdn_prefill_desc* d) {
    if (d == nullptr) return GDN_ERR_INVALID_ARG;
    int st;
    if (d->T_total == 0) {
        // no token rows: the token tensors may have no storage (null pointers)
        alignas(16) static const float kNoRows[4] = {};
        gdn_prefill_desc e = *d;
        e.q = e.k = e.v = kNoRows;
        e.out = const_cast<float*>(kNoRows);            // only validated, never written
        e.g = e.beta = kNoRows;
        e.conv_x = nullptr;
        st = check_common(&e);
        if (st == GDN_OK && d->conv_state_out != nullptr && (d->conv_kernel < 2 || d->conv_kernel > 8))
            st = GDN_ERR_UNSUPPORTED;
    } else {
        st = check_common(d);
    }
    if (st != GDN_OK) return st;
    if (d->chunk < 1 || d->chunk > gdn::kMaxChunk) return GDN_ERR_CHUNK;
    if (d->cu_seqlens == nullptr) return GDN_ERR_INVALID_ARG;
    if (d->conv_x != nullptr) {
        if (d->T_total < 0) return GDN_ERR_INVALID_ARG;
        const size_t need = conv_workspace(d);
        if (need > 0) {
            if (d->workspace == nullptr || d->workspace_bytes < need) return GDN_ERR_WORKSPACE;
            if ((reinterpret_cast<uintptr_t>(d->workspace) & 255u) != 0) return GDN_ERR_WORKSPACE;
        }
    }
    return GDN_OK;
}

// A batch without a token (T_total == 0): every sequence keeps its states
// (an empty sequence returns its incoming state), by stream-ordered device
// copies or, without an incoming state, zero fills.  No kernel runs.
int empty_prefill(const gdn_prefill_desc* d, cudaStream_t s) {
    const size_t state_bytes = size_t(d->B) * size_t(d->Hv) * size_t(d->dk) * size_t(d->dv) * sizeof(float);
    cudaError_t e = cudaSuccess;
    if (d->state_out != nullptr && d->state_out != d->state_in)
        e = d->state_in != nullptr
                ? cudaMemcpyAsync(d->state_out, d->state_in, state_bytes, cudaMemcpyDeviceToDevice, s)
                : cudaMemsetAsync(d->state_out, 0, state_bytes, s);
    if (e == cudaSuccess && d->conv_state_out != nullptr && d->conv_state_out != d->conv_state_in) {
        const size_t conv_bytes = size_t(d->B) * size_t(conv_channels(d)) * size_t(d->conv_kernel - 1) * sizeof(float);
        e = d->conv_state_in != nullptr
                ? cudaMemcpyAsync(d->conv_state_out, d->conv_state_in, conv_bytes, cudaMemcpyDeviceToDevice, s)
                : cudaMemsetAsync(d->conv_state_out, 0, conv_bytes, s);
    }
    return cuda_status(e);
}

}  // namespace

namespace gdn {
size_t prefill_required_workspace(const gdn_prefill_desc* d) { return conv_workspace(d); }
}  // namespace gdn

extern "C" {

void gdn_prefill_desc_init(gdn_prefill_desc* d) {
    if (d == nullptr) return;
    std::memset(d, 0, sizeof(*d));
    d->dtype = GDN_BF16;
    d->chunk = gdn::kMaxChunk;
    d->T_total = -1;
    d->conv_kernel = 4;
    d->conv_act = GDN_ACT_NONE;
    d->use_qk_l2norm = 1;
    d->l2_eps = 1e-6f;
    d->q_scale = 1.f;
}

size_t gdn_workspace_bytes(const gdn_prefill_desc* d) {
    // Only the shape fields matter here; tensor pointers may still be unset.
    if (d == nullptr) return size_t(-1);
    if (d->dtype != GDN_BF16 && d->dtype != GDN_FP32) return size_t(-1);
    if (d->B < 0 || d->Hk <= 0 || d->Hv <= 0 || d->Hv % d->Hk != 0) return size_t(-1);
    if (!head_dim_ok(d->dk) || !head_dim_ok(d->dv)) return size_t(-1);
    if (d->conv_x != nullptr && d->T_total < 0) return size_t(-1);
    if (d->chunk < 1 || d->chunk > gdn::kMaxChunk) return size_t(-1);
    return workspace_needed(d);
}

int gdn_prefill_ex(const gdn_prefill_desc* d, gdn_stream_t stream) {
    const int st = check_prefill(d);
    if (st != GDN_OK) return st;
    if (d->B == 0) return GDN_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (d->T_total == 0) return empty_prefill(d, s);

    gdn::ChunkParams p{};
    p.g = d->g;
    p.beta = d->beta;
    p.state_in = d->state_in;
    p.state_out = d->state_out;
    p.out = d->out;
    p.cu = d->cu_seqlens;
    p.t_cap = d->T_total >= 0 ? d->T_total : INT64_MAX;
    p.B = d->B;
    p.Hk = d->Hk;
    p.Hv = d->Hv;
    p.dk = d->dk;
    p.dv = d->dv;
    p.chunk = d->chunk;
    p.l2norm = d->use_qk_l2norm;
    p.eps = d->l2_eps;
    p.q_scale = d->q_scale;
    {
        // segment-parallel scan when chosen and the workspace holds its maps;
        // split preparation when on and the workspace also holds the records
        const int sc = segment_chunks(d);
        const size_t conv_bytes = conv_workspace(d);
        const size_t seg_bytes = segment_workspace(d, sc);
        const size_t prep_bytes = prep_workspace(d);
        if (sc > 0 && d->workspace != nullptr && d->workspace_bytes >= conv_bytes + seg_bytes) {
            const int64_t seg_tokens = int64_t(sc) * d->chunk;
            p.seg_chunks = sc;
            p.seg_ws = reinterpret_cast<float*>(static_cast<char*>(d->workspace) + conv_bytes);
            p.seg_slots = segment_slots(d, sc);
            p.seg_max = int((d->T_total + seg_tokens - 1) / seg_tokens);
            seg_out_plan(int64_t(d->Hv) * d->B, p.seg_max, sc, &p.seg_final_cta, &p.seg_groups,
                         p.seg_max - 1 <= gdn::kSegTable ? p.seg_gstart : nullptr);
            p.g_out = static_cast<char*>(d->workspace) + conv_bytes + segment_map_bytes(d, sc);
        }
        if (prep_bytes > 0 && d->workspace != nullptr &&
            d->workspace_bytes >= conv_bytes + seg_bytes + prep_bytes) {
            p.prep_ws = static_cast<uint8_t*>(d->workspace) + conv_bytes + seg_bytes;
            p.prep_slots = prep_slots(d);
        }
    }

    if (d->conv_x != nullptr) {
        const int64_t C = conv_channels(d);
        gdn::ConvParams c{};
        c.x = d->conv_x;
        c.w = d->conv_w;
        c.state_in = d->conv_state_in;
        c.state_out = d->conv_state_out;
        c.y = d->workspace;
        c.cu = d->cu_seqlens;
        c.T = d->T_total;
        c.B = d->B;
        c.C = int(C);
        c.K = d->conv_kernel;
        c.act = d->conv_act;
        int rc = cuda_status(gdn::launch_conv(c, d->dtype, s));
        if (rc != GDN_OK) return rc;
        const size_t es = elem_size(d->dtype);
        const char* y = static_cast<const char*>(d->workspace);
        p.q = y;
        p.k = y + size_t(d->Hk) * d->dk * es;
        p.v = y + size_t(2) * d->Hk * d->dk * es;
        p.q_stride = p.k_stride = p.v_stride = C;
        rc = cuda_status(gdn::tc_supported(p, d->dtype) ? gdn::launch_chunk_tc(p, s)
                                                        : gdn::launch_chunk_simt(p, d->dtype, s));
        if (rc != GDN_OK) return rc;
        // The chunk kernels read the workspace, not x, so the conv state can be
        // advanced last; this also keeps an aliased in/out conv state safe.
        return cuda_status(gdn::launch_conv_state(c, d->dtype, s));
    }
    p.q = d->q;
    p.k = d->k;
    p.v = d->v;
    p.q_stride = p.k_stride = int64_t(d->Hk) * d->dk;
    p.v_stride = int64_t(d->Hv) * d->dv;
    return cuda_status(gdn::tc_supported(p, d->dtype) ? gdn::launch_chunk_tc(p, s)
                                                      : gdn::launch_chunk_simt(p, d->dtype, s));
}

int gdn_prefill(const void* q, const void* k, const void* v, const float* g, const float* beta,
                const float* state_in, float* state_out, void* out, const int32_t* cu_seqlens,
                int B, int Hk, int Hv, int dk, int dv, int chunk, gdn_stream_t stream) {
    gdn_prefill_desc d;
    gdn_prefill_desc_init(&d);
    d.q = q;
    d.k = k;
    d.v = v;
    d.g = g;
    d.beta = beta;
    d.state_in = state_in;
    d.state_out = state_out;
    d.out = out;
    d.cu_seqlens = cu_seqlens;
    d.B = B;
    d.Hk = Hk;
    d.Hv = Hv;
    d.dk = dk;
    d.dv = dv;
    d.chunk = chunk;
    return gdn_prefill_ex(&d, stream);
}

int gdn_step_ex(const gdn_prefill_desc* d, gdn_stream_t stream) {
    const int st = check_common(d);
    if (st != GDN_OK) return st;
    if (d->cu_seqlens != nullptr) return GDN_ERR_INVALID_ARG;
    if (d->B == 0) return GDN_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    gdn::StepParams p{};
    p.q = d->q;
    p.k = d->k;
    p.v = d->v;
    p.conv_x = d->conv_x;
    p.conv_w = d->conv_w;
    p.conv_state_in = d->conv_state_in;
    p.conv_state_out = d->conv_state_out;
    p.conv_K = d->conv_kernel;
    p.conv_act = d->conv_act;
    p.g = d->g;
    p.beta = d->beta;
    p.state_in = d->state_in;
    p.state_out = d->state_out;
    p.out = d->out;
    p.B = d->B;
    p.Hk = d->Hk;
    p.Hv = d->Hv;
    p.dk = d->dk;
    p.dv = d->dv;
    p.l2norm = d->use_qk_l2norm;
    p.eps = d->l2_eps;
    p.q_scale = d->q_scale;
    int rc = cuda_status(gdn::launch_step(p, d->dtype, s));
    if (rc != GDN_OK) return rc;
    return cuda_status(gdn::launch_step_conv_state(p, d->dtype, s));
}

int gdn_step(const void* q, const void* k, const void* v, const float* g, const float* beta,
             float* state, void* out, int B, int Hk, int Hv, int dk, int dv,
             gdn_stream_t stream) {
    gdn_prefill_desc d;
    gdn_prefill_desc_init(&d);
    d.q = q;
    d.k = k;
    d.v = v;
    d.g = g;
    d.beta = beta;
    d.state_in = state;
    d.state_out = state;
    d.out = out;
    d.B = B;
    d.Hk = Hk;
    d.Hv = Hv;
    d.dk = dk;
    d.dv = dv;
    return gdn_step_ex(&d, stream);
}

int gdn_prefill_plan(const gdn_prefill_desc* d, const char** names, int max_names) {
    const int st = check_prefill(d);
    if (st != GDN_OK) return -st;
    if (d->B == 0 || d->T_total == 0) return 0;      // nothing, or stream-ordered copies only
    const char* plan[6];
    int n = 0;
    gdn::ChunkParams p{};
    p.Hk = d->Hk;
    p.Hv = d->Hv;
    p.dk = d->dk;
    p.dv = d->dv;
    p.chunk = d->chunk;
    if (d->conv_x != nullptr && d->T_total > 0) plan[n++] = "conv_kernel";
    const bool tc = gdn::tc_supported(p, d->dtype);
    const int sc = tc ? segment_chunks(d) : 0;
    const size_t prep_bytes = tc ? prep_workspace(d) : 0;
    const bool records = prep_bytes > 0 && d->workspace != nullptr &&
                         d->workspace_bytes >= conv_workspace(d) + segment_workspace(d, sc) + prep_bytes;
    if (records) plan[n++] = "chunk_prep_kernel";
    plan[n++] = !tc ? "chunk_simt_kernel" : (records ? "chunk_state_kernel" : gdn::kTcKernelName);
    if (sc > 0 && d->workspace != nullptr &&
        d->workspace_bytes >= conv_workspace(d) + segment_workspace(d, sc)) {
        const int64_t seg_tokens = int64_t(sc) * d->chunk;
        const int64_t seg_max = (d->T_total + seg_tokens - 1) / seg_tokens;
        if (seg_max >= 2) plan[n++] = "seg_out_kernel";
    }
    if (d->conv_x != nullptr && d->conv_state_out != nullptr) plan[n++] = "conv_state_kernel";
    for (int i = 0; i < n && i < max_names; ++i)
        if (names != nullptr) names[i] = plan[i];
    return n;
}

const char* gdn_status_string(int status) {
    switch (status) {
        case GDN_OK: return "ok";
        case GDN_ERR_INVALID_ARG: return "invalid argument (null pointer, negative size or bad layout)";
        case GDN_ERR_CHUNK: return "chunk must be in 1..64";
        case GDN_ERR_UNSUPPORTED: return "unsupported shape or option (dk, dv in {16,32,64,128}; Hv % Hk == 0)";
        case GDN_ERR_ALIGN: return "tensor pointer not 16-byte aligned";
        case GDN_ERR_CUDA: return "CUDA launch failed";
        case GDN_ERR_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
        case GDN_ERR_TOO_LARGE: return "size beyond what this entry point supports";
        default: return "unknown status";
    }
}

size_t gdn_scan_workspace_bytes(int C, int64_t T_total) {
    if (C <= 0 || T_total < 0) return size_t(-1);
    return gdn::scan_workspace_bytes(C, T_total);
}

int gdn_scan_rows(const float* a, const float* b, const float* h_in, float* h_out, float* h_rows,
                  const int32_t* cu_seqlens, int B, int C, int64_t T_total, void* workspace,
                  size_t workspace_bytes, gdn_stream_t stream) {
    if (B < 0 || C <= 0 || T_total < 0) return GDN_ERR_INVALID_ARG;
    if (B == 0) return T_total == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
    if (h_out == nullptr || cu_seqlens == nullptr) return GDN_ERR_INVALID_ARG;
    if (T_total > 0 && (a == nullptr || b == nullptr || h_rows == nullptr)) return GDN_ERR_INVALID_ARG;
    if (C % 4 != 0) return GDN_ERR_UNSUPPORTED;
    if (!aligned16(a) || !aligned16(b) || !aligned16(h_rows)) return GDN_ERR_ALIGN;
    const int64_t tiles = ((T_total + gdn::rows::kScanRows - 1) / gdn::rows::kScanRows) * ((int64_t(C) + gdn::rows::kCols - 1) / gdn::rows::kCols);
    if (tiles > INT32_MAX) return GDN_ERR_TOO_LARGE;
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
        workspace_bytes < gdn::scan_workspace_bytes(C, T_total))
        return GDN_ERR_WORKSPACE;
    gdn::ScanParams p{};
    p.a = a;
    p.b = b;
    p.h_in = h_in;
    p.h_out = h_out;
    p.h_rows = h_rows;
    p.cu = cu_seqlens;
    p.T = T_total;
    p.B = B;
    p.C = C;
    gdn::scan_bind_workspace(p, workspace);
    return cuda_status(gdn::launch_scan_rows(p, static_cast<cudaStream_t>(stream)));
}

size_t gdn_wkv_workspace_bytes(int C, int64_t T_total) {
    if (C <= 0 || T_total < 0) return size_t(-1);
    return gdn::wkv_workspace_bytes(C, T_total);
}

int gdn_wkv_rows(const float* k, const float* v, const float* w, const float* u,
                 const float* state_in, float* state_out, float* wkv, const int32_t* cu_seqlens,
                 int B, int C, int64_t T_total, void* workspace, size_t workspace_bytes,
                 gdn_stream_t stream) {
    if (B < 0 || C <= 0 || T_total < 0) return GDN_ERR_INVALID_ARG;
    if (B == 0) return T_total == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
    if (state_out == nullptr || cu_seqlens == nullptr || w == nullptr || u == nullptr)
        return GDN_ERR_INVALID_ARG;
    if (T_total > 0 && (k == nullptr || v == nullptr || wkv == nullptr)) return GDN_ERR_INVALID_ARG;
    if (C % 4 != 0) return GDN_ERR_UNSUPPORTED;
    if (!aligned16(k) || !aligned16(v) || !aligned16(wkv)) return GDN_ERR_ALIGN;
    const int64_t tiles = ((T_total + gdn::rows::kWkvRows - 1) / gdn::rows::kWkvRows) * ((int64_t(C) + gdn::rows::kCols - 1) / gdn::rows::kCols);
    if (tiles > INT32_MAX) return GDN_ERR_TOO_LARGE;
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
        workspace_bytes < gdn::wkv_workspace_bytes(C, T_total))
        return GDN_ERR_WORKSPACE;
    gdn::WkvParams p{};
    p.k = k;
    p.v = v;
    p.w = w;
    p.u = u;
    p.state_in = state_in;
    p.state_out = state_out;
    p.wkv = wkv;
    p.cu = cu_seqlens;
    p.T = T_total;
    p.B = B;
    p.C = C;
    gdn::wkv_bind_workspace(p, workspace);
    return cuda_status(gdn::launch_wkv_rows(p, static_cast<cudaStream_t>(stream)));
}

int gdn_attn_rows(const void* q, const void* k, const void* v, void* k_cache, void* v_cache,
                  const int32_t* cache_len, void* o, const int32_t* cu_seqlens, int B, int Hq, int Hkv,
                  int head_dim, int cache_capacity, int64_t T_total, float scale, gdn_stream_t stream) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || T_total < 0 || cache_capacity <= 0 || !(scale >= 0.f))
        return GDN_ERR_INVALID_ARG;
    if (head_dim != 128 || Hq % Hkv != 0) return GDN_ERR_UNSUPPORTED;
    if (B == 0) return T_total == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
    if (B > 65535 || Hq > 65535 || T_total > INT32_MAX ||
        int64_t(B) * Hkv * cache_capacity > INT32_MAX)
        return GDN_ERR_TOO_LARGE;
    if (cu_seqlens == nullptr || cache_len == nullptr || k_cache == nullptr || v_cache == nullptr)
        return GDN_ERR_INVALID_ARG;
    if (T_total > 0 && (q == nullptr || k == nullptr || v == nullptr || o == nullptr))
        return GDN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(k_cache) ||
        !aligned16(v_cache))
        return GDN_ERR_ALIGN;
    gdn::AttnParams p{};
    p.q = q;
    p.k = k;
    p.v = v;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.o = o;
    p.cu = cu_seqlens;
    p.cache_len = cache_len;
    p.T = T_total;
    p.max_len = T_total;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.cap = cache_capacity;
    p.scale = scale > 0.f ? scale : 0.08838834764831845f;   // 1 / sqrt(128)
    return cuda_status(gdn::launch_attn_rows(p, static_cast<cudaStream_t>(stream)));
}

long long gdn_wait_timeouts(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    const int a = gdn::tc_read_timeouts(), b = gdn::scan_read_timeouts(), c = gdn::wkv_read_timeouts(),
              d = gdn::attn_read_timeouts();
    if (a < 0 || b < 0 || c < 0 || d < 0) return -1;
    return (long long)a + b + c + d;
}

int gdn_last_cuda_error(void) { return g_last_cuda_error; }

int gdn_version(void) { return 100; }

}  // extern "C"
