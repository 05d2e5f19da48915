// The forward kernels with fp16 MMA operands (fp16 v, and fp16 or fp32 q/k):
// the same source as st_fwd.cu, compiled as its own translation unit.
#define ST_OPERAND_F16 true
#include "st_fwd.cu"
