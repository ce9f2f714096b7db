// Backward kernels (filled in below the forward path).
#include "fa_internal.h"
