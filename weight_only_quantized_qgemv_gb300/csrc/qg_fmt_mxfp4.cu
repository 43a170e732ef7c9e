// Streaming kernels and launchers for the mxfp4 weight format.
#include "qg_device.cuh"
#define QG_FMT ::qg::FMT_MXFP4_G32
#define QG_NAME mxfp4
#include "qg_fmt_impl.cuh"
