// Streaming kernels and launchers for the int4 weight format.
#include "qg_device.cuh"
#define QG_FMT ::qg::FMT_INT4_G
#define QG_NAME int4
#include "qg_fmt_impl.cuh"
