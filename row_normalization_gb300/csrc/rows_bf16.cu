// rows_bf16.cu -- the row-normalization kernels instantiated for bf16.
#include "row_kernels.cuh"

namespace rn {

int rows_run_bf16(const RowCall &c) { return rows_run<Bf16>(c); }

int rows_status_bf16(unsigned int *out, int clear) { return rows_status_word(out, clear); }

int rows_select_schedule(int op, int64_t M, int64_t N) { return rows_select(op, M, N); }

}  // namespace rn
