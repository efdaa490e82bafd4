// od_bwd.cuh -- backward kernels (placeholder until the tcgen05 backward lands).
#pragma once
#include <cuda_runtime.h>
#include <cstddef>

namespace od {

struct BwdArgs {
  int is_time;
  const void *q, *k, *v, *o, *dout;
  const float* lse;
  void *dq, *dk, *dv;
  float *dq_f32, *dk_f32, *dv_f32;
  int B, T, S, Hq, Hkv, D, agent, window;
  float scale;
  void* workspace;
  size_t workspace_bytes;
  cudaStream_t stream;
  unsigned int* status;
  int num_sms;
};

inline cudaError_t bwd_setup() { return cudaSuccess; }
inline size_t bwd_workspace_bytes(int B, int T, int S, int Hq, int D) {
  return size_t(B) * T * S * Hq * (size_t(D) + 1) * 4;
}
// returns 0 on success, 2 when unsupported, 3 on a CUDA error
inline int launch_bwd(const BwdArgs&) { return 2; }

}  // namespace od
