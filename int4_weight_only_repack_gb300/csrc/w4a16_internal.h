// Internal declarations shared by the library's translation units (host side).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/w4a16.h"

namespace w4 {

// Launchers. Arguments are validated by the C-ABI layer before these run.
cudaError_t launch_awq_to_std(const int32_t* qweight, int32_t* qw_out, int K, int N,
                              cudaStream_t s);
cudaError_t launch_to_tile(const int32_t* src, int src_is_awq, const int32_t* perm,
                           int32_t* qw_out, int K, int N, cudaStream_t s);
cudaError_t launch_std_rows_permuted(const int32_t* src, const int32_t* perm, int32_t* qw_out,
                                     int K, int N, cudaStream_t s);
cudaError_t launch_meta(const int32_t* qzeros, int zeros_are_awq, const void* scales,
                        int32_t* zeros_out, void* scales_out, int G, int N, cudaStream_t s);
cudaError_t launch_act_order_perm(const int32_t* g_idx, int K, int group, int32_t* perm_out,
                                  int32_t* status_out, cudaStream_t s);
// An empty kernel launched in full stream order after the repack kernels: the
// GEMM kernels may read their weights before the kernel just before them on the
// stream has finished (programmatic dependent launch), and this keeps that
// kernel from being one that writes weights.
cudaError_t launch_stream_fence(cudaStream_t s);
cudaError_t launch_dequant(const int32_t* qw, const void* scales, const int32_t* zeros, int K,
                           int N, int group, int bf16, int layout, int out_f32, void* w_out,
                           cudaStream_t s);

struct GemmArgs {
  const void* x;
  const uint32_t* qw;
  const void* scales;
  const uint32_t* zeros;
  const int32_t* perm;
  void* y;
  const void* bias;  // [N] in the activation dtype, or nullptr
  int M, N, K, group;
  int bf16;
  void* workspace;
  size_t workspace_bytes;
  int test_stall = 0;  // w4_test_stalled_gemm: the small-M kernel withholds its weight copies
  // grouped (expert) calls of either kernel (w4a16_moe_gemm): M is the most
  // rows any expert has; expert e's rows are [eoff[e], eoff[e + 1]) of x / y
  const int32_t* eoff = nullptr;
  int num_experts = 1;
  int total_rows = 0;
  size_t qw_estride = 0, s_estride = 0, z_estride = 0;  // words / elements / words per expert
};

// Small-M kernel: M rows processed in chunks of up to 64. An act-order call
// given a workspace of decode_workspace_bytes stages x[:, perm] there once
// (launch_gather_columns) and runs the kernel on the staged rows; without it
// every CTA gathers its own slice of x.
constexpr int DECODE_MAX_M = 64;
cudaError_t launch_decode(const GemmArgs& a, cudaStream_t s);
// The streaming small-M kernel (M <= 8, layers of at most 96 KB of packed
// weights per SM, no grouped call): *launched says whether it took the call;
// when it did not, launch_decode runs the clustered kernel instead.
cudaError_t launch_decode_stream(const GemmArgs& a, cudaStream_t s, bool* launched);
size_t decode_workspace_bytes(int M, int K, bool has_perm);

// xg[m][j] = x[m][perm[j]] for M rows of K (16-byte aligned, K % 64 == 0),
// launched with programmatic stream serialization.
cudaError_t launch_gather_columns(const void* x, const int32_t* perm, void* xg, int M, int K,
                                  cudaStream_t s);

// Which kernel a call runs: the small-M kernel for M <= 16, the tcgen05 kernel
// above that when it supports the shape (N % 32 == 0). Measured on GB300 over
// the Llama-2-70B layers: at M = 32 the small-M kernel (4 token tiles) takes
// 57 / 191 / 178 us (qkv / gate_up / down) against 41 / 193 / 91 us for the
// tcgen05 kernel at M = 64 with K split across otherwise idle SMs; at M = 16
// the small-M kernel is still ahead on qkv and gate_up.
bool use_prefill(int M, int N, int K, int sm_count);

// Large-M tcgen05 kernel (N % 32 == 0; w4a16_gemm routes M > 16 here).
// Act-order calls gather x[:, perm] into the workspace first. Grouped calls
// (GemmArgs::eoff set) walk every expert's output tiles in one launch.
bool prefill_supported(int M, int N, int K);
// Whether the large-M kernel takes a grouped (MoE) call of this shape.
bool grouped_prefill_supported(int N, int K, int num_experts);
size_t prefill_workspace_bytes(int M, int K, bool has_perm);
// Further workspace bytes the tcgen05 kernel uses, when given, for the fp32
// partials of its split tiles (0 when it would not split, or when no device
// is current).
size_t prefill_split_workspace_bytes(int M, int N, int K);
// The planner's choice for an ungrouped call on sm_count SMs: rows per tile,
// output tiles, split tiles and K slices of each (out[4]).
void prefill_plan_query(int M, int N, int K, int sm_count, int* out);
cudaError_t launch_prefill(const GemmArgs& a, cudaStream_t s);

// INT4 weights x FP8 activations (w4a8_gemm): workspace bytes for M x K
// activations, and the launch (activation quantisation, then the tcgen05
// kind::f8f6f4 GEMM; group is 128 or K).
size_t w4a8_workspace_bytes(int M, int K);
cudaError_t launch_w4a8(const void* x, const uint32_t* qw, const void* scales,
                        const uint32_t* zeros, void* y, int M, int N, int K, int group, int bf16,
                        void* workspace, cudaStream_t stream);

// Device address and size of the static scratch array of w4a16_gemm_noalloc
// (looked up once per device, with that device current).
cudaError_t noalloc_scratch(void** out, size_t* bytes);

// The device status word the kernels raise on a timed-out wait, and its device
// address (looked up once per device) for the kernels of other translation
// units, which take it as a parameter.
cudaError_t read_device_status(int* out, int clear);
cudaError_t device_status_ptr(int** out);

// cuTensorMapEncodeTiled from the driver (looked up once), and a map over TILE
// words viewed as [column group][k-atom][tile in group][word] (NG column
// groups) whose box is box_tiles tiles x box_atoms k-atoms x box_groups groups.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
bool encode_tile_box(CUtensorMap* map, const void* qw, int K, uint64_t NG, uint32_t box_tiles,
                     uint32_t box_atoms, uint32_t box_groups);

// Device properties cached per device.
struct DeviceInfo {
  int sm_count;
  int major, minor;
  int max_smem_optin;
  int smem_per_sm;
};
cudaError_t device_info(DeviceInfo* out);

}  // namespace w4
