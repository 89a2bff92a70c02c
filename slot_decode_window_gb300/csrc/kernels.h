// Host-side launchers of the window kernels.
#pragma once
#include "common.cuh"

namespace strata {

constexpr int kRouterCols = 512;  // columns per router partial-logit chunk

// Shared-memory plan of the window kernel for one layer shape.  grid: the
// CTAs a decoder stack launches with (its dense phases are cut for the task
// width they run at there), or 0 for a plain window.
KernelCfg window_cfg(const LayerDev& L, int max_rows, int smem_limit, int grid);
// The same with the warp-streamed path (C.direct) where it is the faster one
// and the shape allows it.
KernelCfg window_cfg_direct(const LayerDev& L, int max_rows, int smem_limit);
cudaError_t window_set_attrs(int bits, int direct, int smem_bytes);
// CTAs of the window kernel that one SM holds (0 if it does not fit).
int window_blocks_per_sm(int bits, int direct, int smem_bytes);
// One window: router, grouping, gate/up, down and combine in one cooperative launch.
cudaError_t launch_window(const LayerDev& L, const WindowBufs& W, const KernelCfg& C, int grid, cudaStream_t s);

// A window through n decoder layers (dense q/k/v/o + MoE) in one cooperative
// launch; layers is a device array of n LayerDev.
cudaError_t stack_set_attrs(int bits, int smem_bytes);
int stack_blocks_per_sm(int bits, int smem_bytes);
cudaError_t launch_stack(const LayerDev* layers, int n_layers, int bits, const WindowBufs& W, const KernelCfg& C,
                         int grid, const float* x, float* y, float* ybuf, float* q_all, float* k_all,
                         cudaStream_t s);

// The output head of a window: RMSNorm, the head GEMV over V rows (L.qkv the
// packed head matrix, L.dq = V, W.q_out the logits [T][V]), each row's token
// and each slot's proposal check, in one cooperative launch.
KernelCfg head_cfg(int d, int bits, int max_rows, int smem_limit);
cudaError_t head_set_attrs(int bits, int smem_bytes);
int head_blocks_per_sm(int bits, int smem_bytes);
cudaError_t launch_head(const LayerDev& L, const WindowBufs& W, const KernelCfg& C, const HeadArgs& H, int grid,
                        cudaStream_t s);

// The adaptive tier's round that is due, if any, in a one-CTA launch.
cudaError_t launch_tier_round(const TierDev& Tr, int E, cudaStream_t s);

// Repack one canonical block-quantized matrix stack into the tile format.
cudaError_t launch_repack(const uint8_t* codes, const uint16_t* scale, const uint16_t* mn, int n, int rows, int K,
                          int bits, uint8_t* out, cudaStream_t s);
long long packed_bytes(int n, int rows, int K, int bits);
PackedMat packed_desc(const uint8_t* base, int rows, int K, int bits);

}  // namespace strata
