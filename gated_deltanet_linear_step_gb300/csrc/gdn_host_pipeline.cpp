// gdn_host_pipeline.cpp - decode steps fed from host memory, with the copies of
// neighbouring steps overlapped with the step's kernel (the C ABI in gdn.h).
//
// Each submit queues one step: the host-to-device copies of its qkv, z, alpha
// and beta into one of two device slots, the decode step on those slots, and
// the device-to-host copy of its y. Three streams carry the three stages and
// events order each slot's reuse:
//
//   copy-in k    waits for  step k - 2       (the slot's inputs are free)
//   step k       waits for  copy-in k, and copy-out k - 2 (the slot's y is free)
//   copy-out k   waits for  step k
//
// so step k + 1's inputs travel while step k computes and step k - 1's y
// comes back. The slots are device memory the caller provides; every copy is
// one cudaMemcpyAsync; steps run in submission order on one stream, so the
// state and conv history advance as they would with direct calls.

#include <cstddef>
#include <cstdint>
#include <new>

#include <cuda_runtime.h>

#include "gdn.h"
#include "gdn_launch.h"

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t n) { return (n + kAlign - 1) / kAlign * kAlign; }

struct SlotSizes {
    size_t qkv, z, gates, y, total;
};

SlotSizes slot_sizes(int B, int L, int T) {
    const size_t rows = static_cast<size_t>(B) * L * T;
    SlotSizes s;
    s.qkv = rows * gdn::kConvChannels * 4;
    s.z = rows * gdn::kValueDim * 4;
    s.gates = rows * gdn::kVHeads * 4;
    s.y = rows * gdn::kValueDim * 4;
    s.total = round_up(s.qkv) + round_up(s.z) + 2 * round_up(s.gates) + round_up(s.y);
    return s;
}

struct Slot {
    float* qkv;
    float* z;
    float* alpha;
    float* beta;
    float* y;
};

}  // namespace

struct gdn_host_pipeline {
    int device;
    int B, L, T;
    SlotSizes sizes;
    Slot slot[2];
    gdn::StepArgs step;  // weights, state, conv history, seq_len; per-step pointers set at submit
    cudaStream_t s_in, s_step, s_out;
    cudaEvent_t ev_in[2], ev_step[2], ev_out[2];
    unsigned long long count;
};

namespace gdn {
gdn_status report_status(gdn_status s, const char* msg);  // gdn_api.cpp
}  // namespace gdn

namespace {

gdn_status fail(gdn_status s, const char* msg) { return gdn::report_status(s, msg); }

// Runs `body` with `dev` as the current device and restores the caller's.
template <class F>
cudaError_t on_device(int dev, F body) {
    int prev = 0;
    cudaError_t e = cudaGetDevice(&prev);
    if (e != cudaSuccess) return e;
    if (prev != dev) {
        e = cudaSetDevice(dev);
        if (e != cudaSuccess) return e;
    }
    const cudaError_t r = body();
    if (prev != dev) {
        e = cudaSetDevice(prev);
        if (r == cudaSuccess && e != cudaSuccess) return e;
    }
    return r;
}

void release(gdn_host_pipeline* p) {
    for (int i = 0; i < 2; ++i) {
        if (p->ev_in[i]) cudaEventDestroy(p->ev_in[i]);
        if (p->ev_step[i]) cudaEventDestroy(p->ev_step[i]);
        if (p->ev_out[i]) cudaEventDestroy(p->ev_out[i]);
    }
    if (p->s_in) cudaStreamDestroy(p->s_in);
    if (p->s_step) cudaStreamDestroy(p->s_step);
    if (p->s_out) cudaStreamDestroy(p->s_out);
}

}  // namespace

extern "C" {

size_t gdn_host_pipeline_slot_bytes(int B, int L, int T) {
    if (B < 1 || L < 1 || L > 65535 || T < 1 || T > gdn::kMaxT) return 0;
    return 2 * slot_sizes(B, L, T).total;
}

gdn_status gdn_host_pipeline_create(gdn_host_pipeline** out, const float* dt, const float* ssm_a,
                                    const float* conv_w, const float* ssm_norm, float* conv_state, float* state,
                                    const int32_t* seq_len, void* slots, size_t slots_bytes, int B, int L, int T,
                                    int device) {
    gdn::report_status(GDN_OK, "");
    if (out == nullptr) return fail(GDN_ERR_NULL, "gdn_host_pipeline_create: out is NULL");
    *out = nullptr;
    const void* need[] = {dt, ssm_a, conv_w, ssm_norm, conv_state, state, slots};
    for (const void* q : need) {
        if (q == nullptr) return fail(GDN_ERR_NULL, "gdn_host_pipeline_create: a device pointer is NULL");
        if ((reinterpret_cast<unsigned long long>(q) & 15ull) != 0)
            return fail(GDN_ERR_ALIGN, "gdn_host_pipeline_create: a device pointer is not 16-byte aligned");
    }
    if (seq_len != nullptr && (reinterpret_cast<unsigned long long>(seq_len) & 3ull) != 0)
        return fail(GDN_ERR_ALIGN, "gdn_host_pipeline_create: seq_len is not 4-byte aligned");
    if (B < 1 || L < 1 || L > 65535 || T < 1 || T > gdn::kMaxT)
        return fail(GDN_ERR_SHAPE, "gdn_host_pipeline_create: B, L or T out of range");
    if ((reinterpret_cast<unsigned long long>(slots) % kAlign) != 0)
        return fail(GDN_ERR_ALIGN, "gdn_host_pipeline_create: slots is not 256-byte aligned");
    const SlotSizes sz = slot_sizes(B, L, T);
    if (slots_bytes < 2 * sz.total)
        return fail(GDN_ERR_SHAPE, "gdn_host_pipeline_create: slots smaller than gdn_host_pipeline_slot_bytes()");

    gdn_host_pipeline* p = new (std::nothrow) gdn_host_pipeline();
    if (p == nullptr) return fail(GDN_ERR_CUDA, "gdn_host_pipeline_create: out of host memory");
    p->device = device;
    p->B = B;
    p->L = L;
    p->T = T;
    p->sizes = sz;
    char* base = static_cast<char*>(slots);
    for (int i = 0; i < 2; ++i) {
        char* c = base + i * sz.total;
        p->slot[i].qkv = reinterpret_cast<float*>(c);
        c += round_up(sz.qkv);
        p->slot[i].z = reinterpret_cast<float*>(c);
        c += round_up(sz.z);
        p->slot[i].alpha = reinterpret_cast<float*>(c);
        c += round_up(sz.gates);
        p->slot[i].beta = reinterpret_cast<float*>(c);
        c += round_up(sz.gates);
        p->slot[i].y = reinterpret_cast<float*>(c);
    }
    gdn::StepArgs& a = p->step;
    a.qkv = nullptr;
    a.z = nullptr;
    a.alpha = nullptr;
    a.beta = nullptr;
    a.dt = dt;
    a.ssm_a = ssm_a;
    a.conv_w = conv_w;
    a.ssm_norm = ssm_norm;
    a.conv_state = conv_state;
    a.state = state;
    a.y = nullptr;
    a.seq_len = seq_len;
    a.B = B;
    a.L = L;
    a.T = T;
    a.flags = 0;
    const cudaError_t e = on_device(device, [&]() -> cudaError_t {
        cudaError_t r = cudaStreamCreateWithFlags(&p->s_in, cudaStreamNonBlocking);
        if (r == cudaSuccess) r = cudaStreamCreateWithFlags(&p->s_step, cudaStreamNonBlocking);
        if (r == cudaSuccess) r = cudaStreamCreateWithFlags(&p->s_out, cudaStreamNonBlocking);
        for (int i = 0; i < 2 && r == cudaSuccess; ++i) {
            r = cudaEventCreateWithFlags(&p->ev_in[i], cudaEventDisableTiming);
            if (r == cudaSuccess) r = cudaEventCreateWithFlags(&p->ev_step[i], cudaEventDisableTiming);
            if (r == cudaSuccess) r = cudaEventCreateWithFlags(&p->ev_out[i], cudaEventDisableTiming);
        }
        return r;
    });
    if (e != cudaSuccess) {
        release(p);
        delete p;
        return fail(GDN_ERR_CUDA, cudaGetErrorString(e));
    }
    *out = p;
    return GDN_OK;
}

gdn_status gdn_host_pipeline_submit(gdn_host_pipeline* p, const float* qkv, const float* z, const float* alpha,
                                    const float* beta, float* y) {
    gdn::report_status(GDN_OK, "");
    if (p == nullptr || qkv == nullptr || z == nullptr || alpha == nullptr || beta == nullptr || y == nullptr)
        return fail(GDN_ERR_NULL, "gdn_host_pipeline_submit: a pointer is NULL");
    const int i = static_cast<int>(p->count & 1ull);
    const bool reuse = p->count >= 2;
    Slot& s = p->slot[i];
    const cudaError_t e = on_device(p->device, [&]() -> cudaError_t {
        cudaError_t r = cudaSuccess;
        if (reuse) r = cudaStreamWaitEvent(p->s_in, p->ev_step[i], 0);
        if (r == cudaSuccess) r = cudaMemcpyAsync(s.qkv, qkv, p->sizes.qkv, cudaMemcpyHostToDevice, p->s_in);
        if (r == cudaSuccess) r = cudaMemcpyAsync(s.z, z, p->sizes.z, cudaMemcpyHostToDevice, p->s_in);
        if (r == cudaSuccess) r = cudaMemcpyAsync(s.alpha, alpha, p->sizes.gates, cudaMemcpyHostToDevice, p->s_in);
        if (r == cudaSuccess) r = cudaMemcpyAsync(s.beta, beta, p->sizes.gates, cudaMemcpyHostToDevice, p->s_in);
        if (r == cudaSuccess) r = cudaEventRecord(p->ev_in[i], p->s_in);
        if (r == cudaSuccess) r = cudaStreamWaitEvent(p->s_step, p->ev_in[i], 0);
        if (r == cudaSuccess && reuse) r = cudaStreamWaitEvent(p->s_step, p->ev_out[i], 0);
        if (r == cudaSuccess) {
            gdn::StepArgs a = p->step;
            a.qkv = s.qkv;
            a.z = s.z;
            a.alpha = s.alpha;
            a.beta = s.beta;
            a.y = s.y;
            r = gdn::launch_decode_step(a, p->s_step);
        }
        if (r == cudaSuccess) r = cudaEventRecord(p->ev_step[i], p->s_step);
        if (r == cudaSuccess) r = cudaStreamWaitEvent(p->s_out, p->ev_step[i], 0);
        if (r == cudaSuccess) r = cudaMemcpyAsync(y, s.y, p->sizes.y, cudaMemcpyDeviceToHost, p->s_out);
        if (r == cudaSuccess) r = cudaEventRecord(p->ev_out[i], p->s_out);
        return r;
    });
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, cudaGetErrorString(e));
    ++p->count;
    return GDN_OK;
}

gdn_status gdn_host_pipeline_synchronize(gdn_host_pipeline* p) {
    gdn::report_status(GDN_OK, "");
    if (p == nullptr) return fail(GDN_ERR_NULL, "gdn_host_pipeline_synchronize: pipeline is NULL");
    const cudaError_t e = on_device(p->device, [&]() -> cudaError_t {
        cudaError_t r = cudaStreamSynchronize(p->s_in);
        if (r == cudaSuccess) r = cudaStreamSynchronize(p->s_step);
        if (r == cudaSuccess) r = cudaStreamSynchronize(p->s_out);
        return r;
    });
    return e == cudaSuccess ? GDN_OK : fail(GDN_ERR_CUDA, cudaGetErrorString(e));
}

void gdn_host_pipeline_destroy(gdn_host_pipeline* p) {
    if (p == nullptr) return;
    (void)on_device(p->device, [&]() -> cudaError_t {
        cudaStreamSynchronize(p->s_in);
        cudaStreamSynchronize(p->s_step);
        cudaStreamSynchronize(p->s_out);
        release(p);
        return cudaSuccess;
    });
    delete p;
}

}  // extern "C"
