// Streaming kernels and launchers for the int8 weight format.
#include "qg_device.cuh"
#define QG_FMT ::qg::FMT_INT8_ROW
#define QG_NAME int8
#include "qg_fmt_impl.cuh"
