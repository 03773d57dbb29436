// Coefficient tables on the host (coeffs.cu): the default table, restart
// windows, and the fp16 range check of the Gram-space backend.
#pragma once

#include <cstddef>
#include <utility>
#include <vector>

namespace dmuon {

// DMuon "API Reference", section YOU_COEFFICIENTS: the default table; rows
// past the fifth repeat the last.
extern const float kYouCoefficients[5][3];

inline const float* coefficient_row(const float* coeffs, int k) {
  return coeffs ? coeffs + 3 * k : kYouCoefficients[k < 4 ? k : 4];
}

// Longest restart window the Gram-space backend runs.  Its fp16 window
// products R Z and Z Q are symmetric only in exact arithmetic (the rounded R
// and Z do not commute) while the kernels store their upper triangle
// mirrored, and that error compounds from step to step of a window.  In an
// emulation of the kernels' roundings (which reproduced the GPU's errors to
// two digits) windows of three steps left 1.5e-2 .. 6.8e-2 relative error on
// inputs whose singular values spread over 164x .. 1e4x (Polar Express and
// printed tables), windows of four or five steps up to 4e-1, and windows of
// at most two steps 1e-3 .. 1.1e-2 on the same inputs.  Restarts do not
// change the result in exact arithmetic, so longer windows are split.
constexpr int kMaxGramWindow = 2;

// Restart windows [start, end) of ns_steps steps: positions outside
// (0, ns_steps) start no window; duplicates collapse; a window longer than
// kMaxGramWindow steps is split into ceil(len / kMaxGramWindow) windows as
// even as possible (longer ones first).
std::vector<std::pair<int, int>> restart_windows(int ns_steps, const std::vector<int>& restarts);

// fp16 range checks of a coefficient table for the direct iteration and
// for the Gram-space backend (see coeffs.cu).  Return true if every buffer
// stays in range for every input; otherwise false with a reason in why
// (why_len bytes, may be null).
bool direct_table_fits(int ns_steps, const float* coeffs, char* why, size_t why_len);
bool gram_table_fits(int ns_steps, const float* coeffs, const std::vector<int>& restarts, char* why,
                     size_t why_len);

}  // namespace dmuon
