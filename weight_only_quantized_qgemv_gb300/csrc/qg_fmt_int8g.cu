// Streaming kernels and launchers for int8 codes with one scale per group.
#include "qg_device.cuh"
#define QG_FMT ::qg::FMT_INT8_G
#define QG_NAME int8g
#include "qg_fmt_impl.cuh"
