// Library-wide entry points: error strings, version, device queries.
#include <stdarg.h>
#include <stdio.h>

#include "common.cuh"

namespace tsv {

static thread_local char g_err[512] = "";

tsv_status fail(tsv_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

void clear_error() { g_err[0] = '\0'; }

tsv_status check_launch(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(TSV_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
    return TSV_OK;
}

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

}  // namespace tsv

extern "C" const char* tsv_last_error(void) { return tsv::g_err; }

extern "C" int tsv_version(void) { return 101; }
