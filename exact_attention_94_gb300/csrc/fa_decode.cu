// Split-KV decode kernels.
#include "fa_internal.h"
