// f16 KV instances of the split kernel (the same set as bf16).
#define PA_INST_KV kKvF16
#define PA_INST_FN split_kernel_f16
#include "pa_inst_bf16.cu"
