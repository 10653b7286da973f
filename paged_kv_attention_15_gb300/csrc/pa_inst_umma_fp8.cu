// fp8 (e4m3fn) instances of the tcgen05 decode kernel.
#define PA_UMMA_FP8 1
#include "pa_inst_umma.cu"
