// Declarations shared between translation units of libmoe.so (not exported).
#pragma once

#include "moe.h"

namespace moe {

// Launches the bf16 grouped GEMM for the data gradient (grouped_gemm.cu):
//   dA[p, c] = sum_n dC[p, n] * B[e, n, c]   (rows p of expert e)
// with B [E, N, K] read in place (MN-major); rows p >= offsets[E] of dA are
// zeros.  dC bf16 [M_cap, N], dA bf16 [M_cap, K].
moe_status_t dgrad_gemm(const void* dC, const void* B, const int32_t* offsets, int E, int M_cap, int N, int K,
                        void* dA, cudaStream_t stream);

// Launches the grouped GEMM's weight-gradient kernel on CTA pairs (grouped_gemm.cu):
//   dB[e, n, c] = sum_j At_g[n, P_e + j] * Bt_g[c, P_e + j]
// over expert e's zero-padded run [P_e, P_e + 64 * ceil(cnt_e / 64)) of the
// transposed operands At_g bf16 [N, P] and Bt_g bf16 [K, P] (P a multiple of
// 64), where cnt_e = offsets[e + 1] - offsets[e] and P_e the prefix of the
// padded counts.  dB bf16 [E, N, K]; an expert without rows gets zeros.
moe_status_t wgrad_gemm(const void* At_g, const void* Bt_g, int64_t P, const int32_t* offsets, int E,
                        int M_cap, int N, int K, void* dB, cudaStream_t stream);

}  // namespace moe
