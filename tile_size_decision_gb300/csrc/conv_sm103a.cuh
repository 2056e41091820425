// H-tiled implicit-GEMM convolution for sm_103a (declarations).
#pragma once
#include "tiles_internal.h"
