// Fused LM-head front end (tcgen05/TMEM GEMM with a verifier epilogue).
#include "../../include/specverify.h"

extern "C" size_t spec_lmhead_workspace_size(int, int, int, int) { return 256; }

extern "C" sv_status spec_lmhead_verify(const void *, const void *, int, const float *, int, int,
                                        int, float, const int32_t *, const float *, int32_t *,
                                        int32_t *, float *, void *, size_t, void *) {
    return SV_ERR_INVALID;
}
