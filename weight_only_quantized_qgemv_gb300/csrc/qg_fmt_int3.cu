// Streaming kernels and launchers for the int3 weight format.
#include "qg_device.cuh"
#define QG_FMT ::qg::FMT_INT3_G64
#define QG_NAME int3
#include "qg_fmt_impl.cuh"
