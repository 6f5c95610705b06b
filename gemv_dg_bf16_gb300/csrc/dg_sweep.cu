// dg_sweep.cu -- on-device sweep that writes the shape table (filled in below).
#include "dg_internal.h"

extern "C" dg_status dg_sweep(const dg_shape* shapes, int n_shapes, const char* out_path, int reps)
{
    (void)shapes;
    (void)n_shapes;
    (void)out_path;
    (void)reps;
    return DG_ERR_INVALID_ARG;
}
