// ag_gemm.cu -- all-gather + matmul on tcgen05 tensor cores (in progress).
#include "internal.h"
#include "ringcoll.h"

extern "C" int ag_gemm(const void *, size_t, void *, const void *, void *, int, int, int, int, int, void *)
{
    return RC_ERR_UNSUPPORTED;
}
