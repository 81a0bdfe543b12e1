// kvcs_kernels.cuh -- every kernel of the library, for kvcs.cu.
#pragma once

#include "kvcs_bulk.cuh"
#include "kvcs_epilogue.cuh"
#include "kvcs_generic.cuh"
#include "kvcs_write.cuh"
