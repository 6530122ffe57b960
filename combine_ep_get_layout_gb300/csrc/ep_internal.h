// Host-side internals shared by the C ABI (ep_api.cu) and the kernel
// translation units.  Not part of the public interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "ep_gb300.h"

namespace ep {

constexpr int kWarpSize = 32;

// Kernels are launched with programmatic stream serialization: each may be
// scheduled while the kernel ahead of it drains, and waits (griddep_wait)
// before touching global memory.
constexpr bool kUsePdl = true;

// Properties of the current device, queried once per device.
struct DeviceInfo {
  int device = -1;
  int num_sms = 0;
  size_t max_smem_per_block_optin = 0;
  size_t smem_per_sm = 0;
};

// The current device's properties; nullptr (and a message) on failure.
const DeviceInfo *current_device_info();

// Record a detail message for ep_last_error() and return the status.
ep_status_t fail(ep_status_t status, const char *fmt, ...);
ep_status_t cuda_fail(cudaError_t err, const char *what);

// ---- layout (ep_layout.cu)
size_t layout_workspace_bytes(int num_tokens, int num_experts, int num_ranks);
ep_status_t launch_layout(const int64_t *topk_idx, int num_tokens, int num_topk, int num_experts,
                          int num_ranks, const ep_layout_t &layout, void *workspace,
                          cudaStream_t stream);

// ---- dispatch (ep_dispatch.cu)
struct DispatchArgs {
  const uint16_t *x;
  int num_tokens, hidden, num_topk, num_experts, num_ranks;
  const int64_t *topk_idx;
  const float *topk_weights;
  const int32_t *token_slot;
  uint32_t *error_word;
  bool fp8;
  void *recv_x;
  float *recv_x_scales;
  int32_t *recv_src_idx;
  int32_t *recv_topk_idx;
  float *recv_topk_weights;
  int recv_capacity;
};
ep_status_t launch_dispatch(const DispatchArgs &a, cudaStream_t stream);

// ---- combine (ep_combine.cu)
struct CombineArgs {
  const uint16_t *y;
  int recv_capacity, hidden, num_tokens, num_ranks, num_topk, num_experts;
  const int32_t *token_slot;
  uint32_t *error_word;
  const int64_t *topk_idx;
  const float *topk_weights;
  uint16_t *out;
};
ep_status_t launch_combine(const CombineArgs &a, cudaStream_t stream);

}  // namespace ep
