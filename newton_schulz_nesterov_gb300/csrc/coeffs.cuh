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

// Restart windows [start, end) of ns_steps steps: positions outside
// (0, ns_steps) start no window; duplicates collapse.
std::vector<std::pair<int, int>> restart_windows(int ns_steps, const std::vector<int>& restarts);

// fp16 range check of a coefficient table under the Gram-space backend
// (see coeffs.cu).  Returns true if every buffer stays in range; otherwise
// false with a reason in why (why_len bytes, may be null).
bool gram_table_fits(int ns_steps, const float* coeffs, const std::vector<int>& restarts, char* why,
                     size_t why_len);

}  // namespace dmuon
