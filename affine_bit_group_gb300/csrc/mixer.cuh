// Host launchers of the gdn and atq mixer kernels (mixer.cu).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>

namespace abg {

// gdn: one token for H heads of D (64, 128 or 256) columns, K conv taps
// (2..8); arguments as abg_gdn.  With `pdl` the kernel's blocks may be
// scheduled while the launch before runs; they read every input after it
// has finished.
cudaError_t launch_gdn(const float *x, const float *conv, float *state, const float *a, const float *b,
                       const float *z, const float *A_log, const float *dt_bias, const float *nw, float *S, float *y,
                       float *ysum, int H, int D, int K, float eps, float eps_n, bool pdl, cudaStream_t stream);
// sets the gdn kernel's shared-memory attribute for D (done by launch_gdn too)
cudaError_t prepare_gdn(int D);
// atq: one token for Hq query heads over Hkv key/value heads of D (64, 128 or
// 256) columns at position pos (pos + 1 <= 8192); as abg_atq (Kc and Vc
// 16-byte aligned).  Four launches; with `pdl` the last three start early
// (the third copies its value rows meanwhile).  scratch:
// atq_scratch_bytes(Hq, D, pos) bytes of device memory for the chunk results,
// or null for a per-device buffer shared by all such calls.
size_t atq_scratch_bytes(int Hq, int D, int pos);
// sets the value kernel's shared-memory attribute (done by launch_atq too)
cudaError_t prepare_atq(int Hq, int Hkv, int D);
cudaError_t launch_atq(const float *q, const float *gate, const float *k, const float *v, const float *qn_w,
                       const float *kn_w, const float *cs, const float *sn, float *Kc, float *Vc, float *y,
                       float *ysum, int Hq, int Hkv, int D, int P, int pos, float eps, float *scratch, bool pdl,
                       cudaStream_t stream);
// this unit's device status word (OR-ed into *bits)
cudaError_t mixer_status(unsigned *bits, bool clear);

}  // namespace abg
