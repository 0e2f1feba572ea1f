// Internal interface between the C ABI (gdn_api.cpp) and the CUDA kernels (gdn_step.cu).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace gdn {

// Compiled geometry (header comment of Winery-Strata include/strata/core/layer.hpp;
// q|k|v views of gdn_layer step 4 on src/core/layer.cpp).
constexpr int kHeadDim = 128;
constexpr int kKHeads = 16;
constexpr int kVHeads = 48;
constexpr int kGroup = kVHeads / kKHeads;  // v heads per k head
constexpr int kConvChannels = 10240;
constexpr int kValueDim = kVHeads * kHeadDim;
constexpr int kDConv = 4;
constexpr int kKOffset = kKHeads * kHeadDim;      // 2048
constexpr int kVOffset = 2 * kKHeads * kHeadDim;  // 4096
constexpr int kMaxT = 1024;
constexpr int kThreads = kGroup * kHeadDim;       // 384: one thread per state column of 3 tiles

// Kernel behaviour bits (match GDN_FLAG_* in gdn.h).
constexpr uint32_t kNoStateWrite = 0x1u;
constexpr uint32_t kNoY = 0x2u;
constexpr uint32_t kSiluGate = 0x4u;
constexpr uint32_t kGatesReady = 0x8u;  // alpha holds the log decay, beta holds beta (post-activation)
constexpr uint32_t kTestGiveUp = 0x10u;  // the first wait on a state tile of every CTA gives up (tests the drain)

struct StepArgs {
    const float* qkv;
    const float* z;
    const float* alpha;
    const float* beta;
    const float* dt;
    const float* ssm_a;
    const float* conv_w;
    const float* ssm_norm;
    float* conv_state;
    float* state;
    float* y;
    const int32_t* seq_len;
    int B, L, T;
    uint32_t flags;
};

struct AbArgs {
    const float* x;
    const uint16_t* w_alpha;
    const uint16_t* w_beta;
    const float* dt;
    const float* ssm_a;
    float* gate;
    float* beta;
    int B, L, T, n_embd;
};

struct ProjArgs {
    const float* x;
    const uint16_t* w_qkv;
    const uint16_t* w_gate;
    float* qkv;
    float* z;
    void* workspace;
    int B, L, T, n_embd;
    // Optional (all NULL, or all set): the alpha/beta projections with the gate epilogue.
    const uint16_t* w_alpha = nullptr;
    const uint16_t* w_beta = nullptr;
    const float* dt = nullptr;
    const float* ssm_a = nullptr;
    float* gate = nullptr;
    float* beta = nullptr;
    // Optional: weights packed by launch_pack_proj; then w_qkv, w_gate, w_alpha and
    // w_beta are not read, and gate != NULL selects the alpha/beta tile.
    const void* packed = nullptr;
};

// The weights of the input projections, rearranged once into the blocks the
// tensor cores read (gdn_proj.cu). w_alpha and w_beta may be NULL (zero rows).
struct PackArgs {
    const uint16_t* w_qkv;
    const uint16_t* w_gate;
    const uint16_t* w_alpha;
    const uint16_t* w_beta;
    void* packed;
    int L, n_embd;
};

// Blocking of the input projections: token blocks, rows per block (a multiple
// of 16), 64-wide slices of n_embd, pipeline stages.
struct ProjGeometry {
    int n_tb, n_blk, n_ks, n_stages;
};

ProjGeometry proj_geometry(int B, int T, int n_embd);
size_t proj_workspace_bytes(int B, int L, int T, int n_embd);

// The split of x, then the tensor-core projection (gdn_proj.cu).
cudaError_t launch_in_proj(const ProjArgs& a, cudaStream_t stream);

// Bytes of the packed weights of L layers, and the packing kernel.
size_t proj_pack_bytes(int L, int n_embd);
cudaError_t launch_pack_proj(const PackArgs& a, cudaStream_t stream);

// launch_in_proj with the workspace in the library's static scratch array
// (gdn_proj_noalloc.cu); the caller checks the size against
// proj_static_scratch_bytes().
cudaError_t launch_in_proj_static(const ProjArgs& a, cudaStream_t stream);
size_t proj_static_scratch_bytes();

// Reads and clears the projection kernel's device error word.
cudaError_t read_proj_error(uint32_t* out);

// The fused alpha/beta projections with their gate epilogue on the tensor cores (gdn_ab.cu).
cudaError_t launch_ab_gates(const AbArgs& a, cudaStream_t stream);

// Reads and clears the alpha/beta kernel's device error word.
cudaError_t read_ab_error(uint32_t* out);

// Launches the fused decode step on `stream`, choosing the kernel by T and the
// launch's size (the dispatch rules are in gdn_step.cu). Returns the launch status.
cudaError_t launch_decode_step(const StepArgs& a, cudaStream_t stream);

// The kernels a decode call can run (values as gdn_dispatch_kernel returns them).
enum class DecodeKernel : int { kSingleToken = 1, kClusters = 2, kChunked = 3, kTensorCore = 4 };

// The kernel launch_decode_step would run for B x L x T on the current device.
cudaError_t decode_kernel_for(int B, int L, int T, DecodeKernel* out);

// The single-token kernel (gdn_decode_t1.cu); requires a.T == 1.
cudaError_t launch_decode_t1(const StepArgs& a, cudaStream_t stream);

// Reads and clears the single-token kernel's device error word.
cudaError_t read_t1_error(uint32_t* out);

// The multi-token kernel with the tiles resident in shared memory, in chunks
// of up to 8 tokens (gdn_chunk.cu); requires a.T >= 2.
cudaError_t launch_decode_chunked(const StepArgs& a, cudaStream_t stream);

// Reads and clears the chunked kernel's device error word.
cudaError_t read_chunk_error(uint32_t* out);

// The multi-token kernel in chunks of up to 64 tokens whose contractions run on
// the tensor cores (gdn_window_tc.cu); requires a.T >= 2.
cudaError_t launch_decode_window_tc(const StepArgs& a, cudaStream_t stream);

// Reads and clears the tensor-core window kernel's device error word.
cudaError_t read_window_tc_error(uint32_t* out);

// Synchronises `stream`, then reads and clears the device error words of both kernels.
cudaError_t read_device_error(cudaStream_t stream, uint32_t* out);

}  // namespace gdn
