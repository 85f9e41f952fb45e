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
//   dB[e, n, c] = sum over expert e's rows p of dC[p, n] * A[p, c]
// with dC bf16 [M_cap, N] and A bf16 [M_cap, K] read in place (MN-major), in
// 64-row k-blocks from offsets[e].  An expert's last, partial k-block
// (cnt_e mod 64 rows, cnt_e = offsets[e + 1] - offsets[e]) comes instead from
// rows [64e, 64e + 64) of the tails, zero-padded copies of those rows:
// dC's bf16 [64E, N] followed by A's bf16 [64E, K].  dB bf16 [E, N, K]; an
// expert without rows gets zeros.
moe_status_t wgrad_gemm(const void* dC, const void* A, const void* tails, const int32_t* offsets, int E,
                        int M_cap, int N, int K, void* dB, cudaStream_t stream);

}  // namespace moe
