// Host-side launchers of the window kernels.
#pragma once
#include "common.cuh"

namespace strata {

void launch_router(const LayerDev& L, const WindowBufs& W, float* partial, cudaStream_t s);
int router_partial_floats(int d, int E);

// Expert phases: 0 = gate/up + SwiGLU (writes h fragments), 1 = down + combine.
SmemCfg expert_smem_cfg(const LayerDev& L, int phase, int max_rows, int smem_limit);
cudaError_t expert_set_attrs(int bits, int phase, int smem_bytes);
cudaError_t launch_expert(const LayerDev& L, const WindowBufs& W, const SmemCfg& C, int phase, int grid,
                          cudaStream_t s, bool pdl);

// Repack one canonical block-quantized matrix stack into the tile format.
cudaError_t launch_repack(const uint8_t* codes, const uint16_t* scale, const uint16_t* mn, int n, int rows, int K,
                          int bits, uint8_t* out, cudaStream_t s);
long long packed_bytes(int n, int rows, int K, int bits);
PackedMat packed_desc(const uint8_t* base, int rows, int K, int bits);

}  // namespace strata
