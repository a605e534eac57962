// rows_f16.cu -- the row-normalization kernels instantiated for IEEE fp16.
#include "row_kernels.cuh"

namespace rn {

int rows_run_f16(const RowCall &c) { return rows_run<F16>(c); }

int rows_status_f16(unsigned int *out, int clear) { return rows_status_word(out, clear); }

}  // namespace rn
