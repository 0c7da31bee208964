// Test shim: the clustered decode kernel's unit-ownership rule (kernels.h),
// built with the host compiler.
#include "kernels.h"

extern "C" int shim_cluster_unit_owner_shared(int G, int Ur, int n_cl) {
  return moe::cluster_unit_owner_shared(G, Ur, n_cl);
}
