// Tensor-core engine (tcgen05 / TMEM / TMA, sm_103a).
#include "sg_internal.cuh"

bool tc_supported(const sg_layout *) { return false; }

static sg_status tc_unavailable(const char *fn)
{
    sg_set_error("%s: the tensor-core engine is not available in this build", fn);
    return SG_ERR_UNSUPPORTED;
}

sg_status tc_fwd(sg_layout *, int32_t, const uint16_t *, uint16_t *, uint16_t *,
                 double *, cudaStream_t)
{
    return tc_unavailable("tc_fwd");
}
sg_status tc_dW(sg_layout *, const uint16_t *, int32_t, uint16_t *, cudaStream_t)
{
    return tc_unavailable("tc_dW");
}
sg_status tc_dh(sg_layout *, const uint16_t *, int32_t, const uint16_t *, float *,
                cudaStream_t)
{
    return tc_unavailable("tc_dh");
}
sg_status tc_step(sg_layout *, int32_t, const uint16_t *, uint16_t *, float *,
                  double *, cudaStream_t)
{
    return tc_unavailable("tc_step");
}
