// Prefill-path kernels of libmoe (sm_103a).  Placeholder translation unit.
#include "common.cuh"
#include "internal.h"
#include "kernels.h"
