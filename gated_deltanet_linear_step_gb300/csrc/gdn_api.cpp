// gdn_api.cpp - the C ABI declared in include/gdn.h: argument checks, error
// messages, and the hand-off to the fused kernel in gdn_step.cu.

#include "gdn.h"

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "gdn_launch.h"

static_assert(GDN_HEAD_DIM == gdn::kHeadDim, "geometry mismatch");
static_assert(GDN_K_HEADS == gdn::kKHeads, "geometry mismatch");
static_assert(GDN_V_HEADS == gdn::kVHeads, "geometry mismatch");
static_assert(GDN_CONV_CHANNELS == gdn::kConvChannels, "geometry mismatch");
static_assert(GDN_VALUE_DIM == gdn::kValueDim, "geometry mismatch");
static_assert(GDN_D_CONV == gdn::kDConv, "geometry mismatch");
static_assert(GDN_MAX_T == gdn::kMaxT, "geometry mismatch");
static_assert(GDN_FLAG_NO_STATE_WRITE == gdn::kNoStateWrite && GDN_FLAG_NO_Y == gdn::kNoY &&
                  GDN_FLAG_SILU_GATE == gdn::kSiluGate && GDN_FLAG_GATES_READY == gdn::kGatesReady &&
                  GDN_FLAG_TEST_GIVE_UP == gdn::kTestGiveUp,
              "flag mismatch");

namespace {

thread_local std::string t_last_error;

gdn_status fail(gdn_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return s;
}

struct Span {
    const char* name;
    const void* p;
    unsigned long long bytes;
    bool output;
};

bool overlaps(const Span& a, const Span& b) {
    if (a.p == nullptr || b.p == nullptr || a.bytes == 0 || b.bytes == 0) return false;
    const unsigned long long a0 = reinterpret_cast<unsigned long long>(a.p);
    const unsigned long long b0 = reinterpret_cast<unsigned long long>(b.p);
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// Checks and launches one decode-step call. `state_ro`/`conv_ro` mark the
// states as read only (no alias rule for them as outputs).
gdn_status run(const float* qkv, const float* z, const float* alpha, const float* beta, const float* dt,
               const float* ssm_a, const float* conv_w, const float* ssm_norm, float* conv_state, float* state,
               float* y, const int32_t* seq_len, int B, int L, int T, uint32_t flags, void* stream,
               const char* fn) {
    t_last_error.clear();
    const uint32_t known = gdn::kNoStateWrite | gdn::kNoY | gdn::kSiluGate | gdn::kGatesReady | gdn::kTestGiveUp;
    if (flags & ~known) return fail(GDN_ERR_FLAGS, "%s: unknown flag bits 0x%x", fn, flags & ~known);
    const bool want_y = (flags & gdn::kNoY) == 0;
    const bool write_state = (flags & gdn::kNoStateWrite) == 0;

    const struct {
        const char* name;
        const void* p;
        bool required;
    } ptrs[] = {{"qkv", qkv, true},       {"z", z, want_y},           {"alpha", alpha, true},
                {"beta", beta, true},     {"dt", dt, true},           {"ssm_a", ssm_a, true},
                {"conv_w", conv_w, true}, {"ssm_norm", ssm_norm, want_y}, {"conv_state", conv_state, true},
                {"state", state, true},   {"y", y, want_y}};
    for (const auto& q : ptrs) {
        if (q.required && q.p == nullptr) return fail(GDN_ERR_NULL, "%s: %s is NULL", fn, q.name);
        if (q.p != nullptr && (reinterpret_cast<unsigned long long>(q.p) & 15ull) != 0)
            return fail(GDN_ERR_ALIGN, "%s: %s is not 16-byte aligned", fn, q.name);
    }
    if (seq_len != nullptr && (reinterpret_cast<unsigned long long>(seq_len) & 3ull) != 0)
        return fail(GDN_ERR_ALIGN, "%s: seq_len is not 4-byte aligned", fn);
    if (B < 1 || L < 1) return fail(GDN_ERR_SHAPE, "%s: B=%d and L=%d must be >= 1", fn, B, L);
    if (T < 1 || T > gdn::kMaxT) return fail(GDN_ERR_SHAPE, "%s: T=%d must be in [1, %d]", fn, T, gdn::kMaxT);

    // Byte sizes in 64-bit; B * L tiles of 3 MB must stay addressable.
    const unsigned long long b = static_cast<unsigned long long>(B), l = static_cast<unsigned long long>(L),
                             t = static_cast<unsigned long long>(T);
    if (b * l > (1ull << 40) / (48ull * 65536ull))
        return fail(GDN_ERR_SHAPE, "%s: B*L=%llu is too large", fn, b * l);
    const unsigned long long blt = b * l * t;
    const Span spans[] = {
        {"qkv", qkv, blt * gdn::kConvChannels * 4, false},
        {"z", z, want_y ? blt * gdn::kValueDim * 4 : 0, false},
        {"alpha", alpha, blt * gdn::kVHeads * 4, false},
        {"beta", beta, blt * gdn::kVHeads * 4, false},
        {"dt", dt, l * gdn::kVHeads * 4, false},
        {"ssm_a", ssm_a, l * gdn::kVHeads * 4, false},
        {"conv_w", conv_w, l * gdn::kConvChannels * gdn::kDConv * 4, false},
        {"ssm_norm", ssm_norm, want_y ? l * gdn::kHeadDim * 4 : 0, false},
        {"seq_len", seq_len, seq_len ? b * 4 : 0, false},
        {"conv_state", conv_state, b * l * gdn::kConvChannels * (gdn::kDConv - 1) * 4, write_state},
        {"state", state, b * l * gdn::kVHeads * 65536ull, write_state},
        {"y", y, want_y ? blt * gdn::kValueDim * 4 : 0, want_y},
    };
    const int n = static_cast<int>(sizeof(spans) / sizeof(spans[0]));
    for (int i = 0; i < n; ++i) {
        if (!spans[i].output) continue;
        for (int k = 0; k < n; ++k)
            if (k != i && overlaps(spans[i], spans[k]))
                return fail(GDN_ERR_ALIAS, "%s: output %s overlaps %s", fn, spans[i].name, spans[k].name);
    }

    gdn::StepArgs a;
    a.qkv = qkv;
    a.z = z;
    a.alpha = alpha;
    a.beta = beta;
    a.dt = dt;
    a.ssm_a = ssm_a;
    a.conv_w = conv_w;
    a.ssm_norm = ssm_norm;
    a.conv_state = conv_state;
    a.state = state;
    a.y = y;
    a.seq_len = seq_len;
    a.B = B;
    a.L = L;
    a.T = T;
    a.flags = flags;
    const cudaError_t e = gdn::launch_decode_step(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "%s: CUDA error: %s", fn, cudaGetErrorString(e));
    return GDN_OK;
}

// One input-projection call. The weights are row-major (w_qkv, w_gate, and with the
// gates w_alpha, w_beta) or packed; the gate arguments (dt, ssm_a, gate, beta) come
// all together or not at all; the split of x goes to the caller's workspace or, with
// `scratch`, to the library's static scratch array.
struct ProjCall {
    const char* fn = "";
    const float* x = nullptr;
    const uint16_t* w_qkv = nullptr;
    const uint16_t* w_gate = nullptr;
    const uint16_t* w_alpha = nullptr;
    const uint16_t* w_beta = nullptr;
    const void* packed = nullptr;
    size_t packed_bytes = 0;
    const float* dt = nullptr;
    const float* ssm_a = nullptr;
    float* qkv = nullptr;
    float* z = nullptr;
    float* gate = nullptr;
    float* beta = nullptr;
    void* workspace = nullptr;
    size_t workspace_bytes = 0;
    int B = 0, L = 0, T = 0, n_embd = 0;
    bool with_ab = false;
    bool use_packed = false;
    bool scratch = false;
};

// Checks a projection call and launches it.
gdn_status run_proj(const ProjCall& c, void* stream) {
    const char* fn = c.fn;
    const bool rowmajor = !c.use_packed;
    const struct {
        const char* name;
        const void* p;
        bool required;
    } ptrs[] = {{"x", c.x, true},
                {"w_qkv", c.w_qkv, rowmajor},
                {"w_gate", c.w_gate, rowmajor},
                {"w_alpha", c.w_alpha, rowmajor && c.with_ab},
                {"w_beta", c.w_beta, rowmajor && c.with_ab},
                {"packed", c.packed, c.use_packed},
                {"dt", c.dt, c.with_ab},
                {"ssm_a", c.ssm_a, c.with_ab},
                {"qkv", c.qkv, true},
                {"z", c.z, true},
                {"gate", c.gate, c.with_ab},
                {"beta", c.beta, c.with_ab},
                {"workspace", c.workspace, !c.scratch}};
    for (const auto& q : ptrs) {
        if (!q.required) continue;
        if (q.p == nullptr) return fail(GDN_ERR_NULL, "%s: %s is NULL", fn, q.name);
        if ((reinterpret_cast<unsigned long long>(q.p) & 15ull) != 0)
            return fail(GDN_ERR_ALIGN, "%s: %s is not 16-byte aligned", fn, q.name);
    }
    const int B = c.B, L = c.L, T = c.T, n_embd = c.n_embd;
    if (B < 1 || L < 1 || L > 65535) return fail(GDN_ERR_SHAPE, "%s: B=%d and L=%d out of range", fn, B, L);
    if (T < 1 || T > gdn::kMaxT) return fail(GDN_ERR_SHAPE, "%s: T=%d must be in [1, %d]", fn, T, gdn::kMaxT);
    if (n_embd < 64 || n_embd > 65536 || n_embd % 64 != 0)
        return fail(GDN_ERR_SHAPE, "%s: n_embd=%d must be a multiple of 64 in [64, 65536]", fn, n_embd);
    const unsigned long long b = B, l = L, t = T, e = n_embd;
    if (b * t > (1ull << 30)) return fail(GDN_ERR_SHAPE, "%s: B*T is too large", fn);
    const size_t need = gdn::proj_workspace_bytes(B, L, T, n_embd);
    if (c.scratch && need > gdn::proj_static_scratch_bytes())
        return fail(GDN_ERR_SHAPE, "%s: these sizes need %zu bytes of scratch, the library holds %zu", fn, need,
                    gdn::proj_static_scratch_bytes());
    if (!c.scratch && c.workspace_bytes < need)
        return fail(GDN_ERR_SHAPE, "%s: workspace of %zu bytes, %zu needed", fn, c.workspace_bytes, need);
    const size_t pack = c.use_packed ? gdn::proj_pack_bytes(L, n_embd) : 0;
    if (c.use_packed && c.packed_bytes < pack)
        return fail(GDN_ERR_SHAPE, "%s: packed weights of %zu bytes, %zu needed", fn, c.packed_bytes, pack);
    const unsigned long long ab = c.with_ab ? 1 : 0, rm = rowmajor ? 1 : 0;
    const Span spans[] = {
        {"x", c.x, b * l * t * e * 4, false},
        {"w_qkv", c.w_qkv, rm * l * gdn::kConvChannels * e * 2, false},
        {"w_gate", c.w_gate, rm * l * gdn::kValueDim * e * 2, false},
        {"w_alpha", c.w_alpha, rm * ab * l * gdn::kVHeads * e * 2, false},
        {"w_beta", c.w_beta, rm * ab * l * gdn::kVHeads * e * 2, false},
        {"packed", c.packed, pack, false},
        {"dt", c.dt, ab * l * gdn::kVHeads * 4, false},
        {"ssm_a", c.ssm_a, ab * l * gdn::kVHeads * 4, false},
        {"qkv", c.qkv, b * l * t * gdn::kConvChannels * 4, true},
        {"z", c.z, b * l * t * gdn::kValueDim * 4, true},
        {"gate", c.gate, ab * b * l * t * gdn::kVHeads * 4, true},
        {"beta", c.beta, ab * b * l * t * gdn::kVHeads * 4, true},
        {"workspace", c.workspace, c.scratch ? 0 : need, true},
    };
    const int n = static_cast<int>(sizeof(spans) / sizeof(spans[0]));
    for (int i = 0; i < n; ++i) {
        if (!spans[i].output) continue;
        for (int k = 0; k < n; ++k)
            if (k != i && overlaps(spans[i], spans[k]))
                return fail(GDN_ERR_ALIAS, "%s: output %s overlaps %s", fn, spans[i].name, spans[k].name);
    }
    gdn::ProjArgs a;
    a.x = c.x;
    a.w_qkv = rowmajor ? c.w_qkv : nullptr;
    a.w_gate = rowmajor ? c.w_gate : nullptr;
    a.qkv = c.qkv;
    a.z = c.z;
    a.workspace = c.scratch ? nullptr : c.workspace;
    a.B = B;
    a.L = L;
    a.T = T;
    a.n_embd = n_embd;
    a.packed = c.use_packed ? c.packed : nullptr;
    if (c.with_ab) {
        a.w_alpha = rowmajor ? c.w_alpha : nullptr;
        a.w_beta = rowmajor ? c.w_beta : nullptr;
        a.dt = c.dt;
        a.ssm_a = c.ssm_a;
        a.gate = c.gate;
        a.beta = c.beta;
    }
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t err = c.scratch ? gdn::launch_in_proj_static(a, st) : gdn::launch_in_proj(a, st);
    if (err != cudaSuccess) return fail(GDN_ERR_CUDA, "%s: CUDA error: %s", fn, cudaGetErrorString(err));
    return GDN_OK;
}

}  // namespace

namespace gdn {
// Status reporting for the other host files of the ABI: records the message
// gdn_last_error() returns on this thread (an empty message clears it).
gdn_status report_status(gdn_status s, const char* msg) {
    t_last_error = msg;
    return s;
}
}  // namespace gdn

extern "C" {

gdn_status gdn_decode_step(const float* qkv, const float* z, const float* alpha, const float* beta,
                           const float* dt, const float* ssm_a, const float* conv_w, const float* ssm_norm,
                           float* conv_state, float* state, float* y, int B, int L, int T, void* stream) {
    return run(qkv, z, alpha, beta, dt, ssm_a, conv_w, ssm_norm, conv_state, state, y, nullptr, B, L, T, 0u,
               stream, "gdn_decode_step");
}

gdn_status gdn_decode_step_varlen(const float* qkv, const float* z, const float* alpha, const float* beta,
                                  const float* dt, const float* ssm_a, const float* conv_w,
                                  const float* ssm_norm, float* conv_state, float* state, float* y,
                                  const int32_t* seq_len, int B, int L, int T, void* stream) {
    return run(qkv, z, alpha, beta, dt, ssm_a, conv_w, ssm_norm, conv_state, state, y, seq_len, B, L, T, 0u,
               stream, "gdn_decode_step_varlen");
}

gdn_status gdn_verify_window(const float* qkv, const float* z, const float* alpha, const float* beta,
                             const float* dt, const float* ssm_a, const float* conv_w, const float* ssm_norm,
                             const float* conv_state, const float* state, float* y, const int32_t* seq_len,
                             int B, int L, int T, void* stream) {
    // The kernel only reads state and conv_state under kNoStateWrite.
    return run(qkv, z, alpha, beta, dt, ssm_a, conv_w, ssm_norm, const_cast<float*>(conv_state),
               const_cast<float*>(state), y, seq_len, B, L, T, gdn::kNoStateWrite, stream, "gdn_verify_window");
}

gdn_status gdn_verify_commit(const float* qkv, const float* alpha, const float* beta, const float* dt,
                             const float* ssm_a, const float* conv_w, float* conv_state, float* state,
                             const int32_t* n_keep, int B, int L, int T, void* stream) {
    if (n_keep == nullptr) return fail(GDN_ERR_NULL, "gdn_verify_commit: n_keep is NULL");
    return run(qkv, nullptr, alpha, beta, dt, ssm_a, conv_w, nullptr, conv_state, state, nullptr, n_keep, B, L, T,
               gdn::kNoY, stream, "gdn_verify_commit");
}

gdn_status gdn_decode_step_ex(const float* qkv, const float* z, const float* alpha, const float* beta,
                              const float* dt, const float* ssm_a, const float* conv_w, const float* ssm_norm,
                              float* conv_state, float* state, float* y, const int32_t* seq_len, int B, int L,
                              int T, uint32_t flags, void* stream) {
    return run(qkv, z, alpha, beta, dt, ssm_a, conv_w, ssm_norm, conv_state, state, y, seq_len, B, L, T, flags,
               stream, "gdn_decode_step_ex");
}

gdn_status gdn_ab_gates(const float* x, const uint16_t* w_alpha, const uint16_t* w_beta, const float* dt,
                        const float* ssm_a, float* gate, float* beta, int B, int L, int T, int n_embd, void* stream) {
    t_last_error.clear();
    const char* fn = "gdn_ab_gates";
    const struct {
        const char* name;
        const void* p;
    } ptrs[] = {{"x", x}, {"w_alpha", w_alpha}, {"w_beta", w_beta}, {"dt", dt},
                {"ssm_a", ssm_a}, {"gate", gate}, {"beta", beta}};
    for (const auto& q : ptrs) {
        if (q.p == nullptr) return fail(GDN_ERR_NULL, "%s: %s is NULL", fn, q.name);
        if ((reinterpret_cast<unsigned long long>(q.p) & 15ull) != 0)
            return fail(GDN_ERR_ALIGN, "%s: %s is not 16-byte aligned", fn, q.name);
    }
    if (B < 1 || L < 1 || L > 65535) return fail(GDN_ERR_SHAPE, "%s: B=%d and L=%d out of range", fn, B, L);
    if (T < 1 || T > gdn::kMaxT) return fail(GDN_ERR_SHAPE, "%s: T=%d must be in [1, %d]", fn, T, gdn::kMaxT);
    if (n_embd < 64 || n_embd > 65536 || n_embd % 64 != 0)
        return fail(GDN_ERR_SHAPE, "%s: n_embd=%d must be a multiple of 64 in [64, 65536]", fn, n_embd);
    const unsigned long long b = B, l = L, t = T, e = n_embd;
    if (b * t > (1ull << 30)) return fail(GDN_ERR_SHAPE, "%s: B*T is too large", fn);
    const Span spans[] = {
        {"x", x, b * l * t * e * 4, false},
        {"w_alpha", w_alpha, l * gdn::kVHeads * e * 2, false},
        {"w_beta", w_beta, l * gdn::kVHeads * e * 2, false},
        {"dt", dt, l * gdn::kVHeads * 4, false},
        {"ssm_a", ssm_a, l * gdn::kVHeads * 4, false},
        {"gate", gate, b * l * t * gdn::kVHeads * 4, true},
        {"beta", beta, b * l * t * gdn::kVHeads * 4, true},
    };
    const int n = static_cast<int>(sizeof(spans) / sizeof(spans[0]));
    for (int i = 0; i < n; ++i) {
        if (!spans[i].output) continue;
        for (int k = 0; k < n; ++k)
            if (k != i && overlaps(spans[i], spans[k]))
                return fail(GDN_ERR_ALIAS, "%s: output %s overlaps %s", fn, spans[i].name, spans[k].name);
    }
    gdn::AbArgs a;
    a.x = x;
    a.w_alpha = w_alpha;
    a.w_beta = w_beta;
    a.dt = dt;
    a.ssm_a = ssm_a;
    a.gate = gate;
    a.beta = beta;
    a.B = B;
    a.L = L;
    a.T = T;
    a.n_embd = n_embd;
    const cudaError_t err = gdn::launch_ab_gates(a, static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return fail(GDN_ERR_CUDA, "%s: CUDA error: %s", fn, cudaGetErrorString(err));
    return GDN_OK;
}

size_t gdn_in_proj_workspace_size(int B, int L, int T, int n_embd) {
    if (B < 1 || L < 1 || L > 65535 || T < 1 || T > gdn::kMaxT || n_embd < 64 || n_embd > 65536 || n_embd % 64 != 0)
        return 0;
    if (static_cast<unsigned long long>(B) * T > (1ull << 30)) return 0;
    return gdn::proj_workspace_bytes(B, L, T, n_embd);
}

gdn_status gdn_in_proj(const float* x, const uint16_t* w_qkv, const uint16_t* w_gate, float* qkv, float* z,
                       void* workspace, size_t workspace_bytes, int B, int L, int T, int n_embd, void* stream) {
    t_last_error.clear();
    ProjCall c;
    c.fn = "gdn_in_proj";
    c.x = x;
    c.w_qkv = w_qkv;
    c.w_gate = w_gate;
    c.qkv = qkv;
    c.z = z;
    c.workspace = workspace;
    c.workspace_bytes = workspace_bytes;
    c.B = B;
    c.L = L;
    c.T = T;
    c.n_embd = n_embd;
    return run_proj(c, stream);
}

gdn_status gdn_step_inputs(const float* x, const uint16_t* w_qkv, const uint16_t* w_gate, const uint16_t* w_alpha,
                           const uint16_t* w_beta, const float* dt, const float* ssm_a, float* qkv, float* z,
                           float* gate, float* beta, void* workspace, size_t workspace_bytes, int B, int L, int T,
                           int n_embd, void* stream) {
    t_last_error.clear();
    ProjCall c;
    c.fn = "gdn_step_inputs";
    c.x = x;
    c.w_qkv = w_qkv;
    c.w_gate = w_gate;
    c.w_alpha = w_alpha;
    c.w_beta = w_beta;
    c.dt = dt;
    c.ssm_a = ssm_a;
    c.qkv = qkv;
    c.z = z;
    c.gate = gate;
    c.beta = beta;
    c.workspace = workspace;
    c.workspace_bytes = workspace_bytes;
    c.B = B;
    c.L = L;
    c.T = T;
    c.n_embd = n_embd;
    c.with_ab = true;
    return run_proj(c, stream);
}

gdn_status gdn_in_proj_noalloc(const float* x, const uint16_t* w_qkv, const uint16_t* w_gate, float* qkv, float* z,
                               int B, int L, int T, int n_embd, void* stream) {
    t_last_error.clear();
    ProjCall c;
    c.fn = "gdn_in_proj_noalloc";
    c.x = x;
    c.w_qkv = w_qkv;
    c.w_gate = w_gate;
    c.qkv = qkv;
    c.z = z;
    c.B = B;
    c.L = L;
    c.T = T;
    c.n_embd = n_embd;
    c.scratch = true;
    return run_proj(c, stream);
}

const char* gdn_last_error(void) { return t_last_error.c_str(); }

int gdn_dispatch_kernel(int B, int L, int T) {
    const char* fn = "gdn_dispatch_kernel";
    if (B < 1 || L < 1 || T < 1 || T > gdn::kMaxT) {
        fail(GDN_ERR_SHAPE, "%s: B=%d, L=%d and T=%d must be >= 1 (T <= %d)", fn, B, L, T, gdn::kMaxT);
        return -1;
    }
    gdn::DecodeKernel k;
    const cudaError_t e = gdn::decode_kernel_for(B, L, T, &k);
    if (e != cudaSuccess) {
        fail(GDN_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
        return -1;
    }
    t_last_error.clear();
    return static_cast<int>(k);
}

gdn_status gdn_get_geometry(int32_t out[8]) {
    if (out == nullptr) return fail(GDN_ERR_NULL, "gdn_get_geometry: out is NULL");
    out[0] = gdn::kHeadDim;
    out[1] = gdn::kKHeads;
    out[2] = gdn::kVHeads;
    out[3] = gdn::kConvChannels;
    out[4] = gdn::kValueDim;
    out[5] = gdn::kDConv;
    out[6] = gdn::kMaxT;
    out[7] = gdn::kThreads;
    return GDN_OK;
}

gdn_status gdn_read_device_error(void* stream, uint32_t* out) {
    t_last_error.clear();
    if (out == nullptr) return fail(GDN_ERR_NULL, "gdn_read_device_error: out is NULL");
    const cudaError_t e = gdn::read_device_error(static_cast<cudaStream_t>(stream), out);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "gdn_read_device_error: %s", cudaGetErrorString(e));
    return GDN_OK;
}

size_t gdn_proj_pack_bytes(int L, int n_embd) {
    if (L < 1 || L > 65535 || n_embd < 64 || n_embd > 65536 || n_embd % 64 != 0) return 0;
    return gdn::proj_pack_bytes(L, n_embd);
}

gdn_status gdn_pack_proj_weights(const uint16_t* w_qkv, const uint16_t* w_gate, const uint16_t* w_alpha,
                                 const uint16_t* w_beta, void* packed, size_t packed_bytes, int L, int n_embd,
                                 void* stream) {
    t_last_error.clear();
    const char* fn = "gdn_pack_proj_weights";
    if ((w_alpha == nullptr) != (w_beta == nullptr))
        return fail(GDN_ERR_NULL, "%s: w_alpha and w_beta must both be given or both be NULL", fn);
    const struct {
        const char* name;
        const void* p;
        bool required;
    } ptrs[] = {{"w_qkv", w_qkv, true}, {"w_gate", w_gate, true}, {"packed", packed, true},
                {"w_alpha", w_alpha, w_alpha != nullptr}, {"w_beta", w_beta, w_beta != nullptr}};
    for (const auto& q : ptrs) {
        if (!q.required) continue;
        if (q.p == nullptr) return fail(GDN_ERR_NULL, "%s: %s is NULL", fn, q.name);
        if ((reinterpret_cast<unsigned long long>(q.p) & 15ull) != 0)
            return fail(GDN_ERR_ALIGN, "%s: %s is not 16-byte aligned", fn, q.name);
    }
    if (L < 1 || L > 65535) return fail(GDN_ERR_SHAPE, "%s: L=%d out of range", fn, L);
    if (n_embd < 64 || n_embd > 65536 || n_embd % 64 != 0)
        return fail(GDN_ERR_SHAPE, "%s: n_embd=%d must be a multiple of 64 in [64, 65536]", fn, n_embd);
    const size_t need = gdn::proj_pack_bytes(L, n_embd);
    if (packed_bytes < need)
        return fail(GDN_ERR_SHAPE, "%s: packed buffer of %zu bytes, %zu needed", fn, packed_bytes, need);
    const unsigned long long l = L, e = n_embd;
    const Span out = {"packed", packed, need, true};
    const Span ins[] = {
        {"w_qkv", w_qkv, l * gdn::kConvChannels * e * 2, false},
        {"w_gate", w_gate, l * gdn::kValueDim * e * 2, false},
        {"w_alpha", w_alpha, w_alpha != nullptr ? l * gdn::kVHeads * e * 2 : 0, false},
        {"w_beta", w_beta, w_beta != nullptr ? l * gdn::kVHeads * e * 2 : 0, false},
    };
    for (const Span& in : ins)
        if (overlaps(out, in)) return fail(GDN_ERR_ALIAS, "%s: packed overlaps %s", fn, in.name);
    gdn::PackArgs a;
    a.w_qkv = w_qkv;
    a.w_gate = w_gate;
    a.w_alpha = w_alpha;
    a.w_beta = w_beta;
    a.packed = packed;
    a.L = L;
    a.n_embd = n_embd;
    const cudaError_t err = gdn::launch_pack_proj(a, static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return fail(GDN_ERR_CUDA, "%s: CUDA error: %s", fn, cudaGetErrorString(err));
    return GDN_OK;
}

gdn_status gdn_in_proj_packed(const float* x, const void* packed, size_t packed_bytes, float* qkv, float* z,
                              void* workspace, size_t workspace_bytes, int B, int L, int T, int n_embd,
                              void* stream) {
    t_last_error.clear();
    ProjCall c;
    c.fn = "gdn_in_proj_packed";
    c.x = x;
    c.packed = packed;
    c.packed_bytes = packed_bytes;
    c.qkv = qkv;
    c.z = z;
    c.workspace = workspace;
    c.workspace_bytes = workspace_bytes;
    c.B = B;
    c.L = L;
    c.T = T;
    c.n_embd = n_embd;
    c.use_packed = true;
    return run_proj(c, stream);
}

gdn_status gdn_step_inputs_packed(const float* x, const void* packed, size_t packed_bytes, const float* dt,
                                  const float* ssm_a, float* qkv, float* z, float* gate, float* beta, void* workspace,
                                  size_t workspace_bytes, int B, int L, int T, int n_embd, void* stream) {
    t_last_error.clear();
    ProjCall c;
    c.fn = "gdn_step_inputs_packed";
    c.x = x;
    c.packed = packed;
    c.packed_bytes = packed_bytes;
    c.dt = dt;
    c.ssm_a = ssm_a;
    c.qkv = qkv;
    c.z = z;
    c.gate = gate;
    c.beta = beta;
    c.workspace = workspace;
    c.workspace_bytes = workspace_bytes;
    c.B = B;
    c.L = L;
    c.T = T;
    c.n_embd = n_embd;
    c.with_ab = true;
    c.use_packed = true;
    return run_proj(c, stream);
}

}  // extern "C"
