// Per-row cross-entropy of the drafter's training forward (kernel in sampling.cu).
#pragma once

#include "launch.h"

namespace dfl {

// out[i*(B-1) + k-1] = -log softmax(logits of row (first_seq + i)*B + k)[labels[i*(B-1) + k-1]]
// for i < n_seqs, k = 1 .. B-1 (fp32 logits, row stride V).
void row_nll(const Launch& L, const float* logits, int V, int B, int first_seq, int n_seqs, const int* labels,
             float* out);

}  // namespace dfl
