// abi.cu -- status names and version of libspecverify.
#include "common.cuh"

SPEC_API const char *spec_strerror(int status) {
    switch (status) {
        case SPEC_OK: return "ok";
        case SPEC_ERR_NULL: return "a required pointer is NULL";
        case SPEC_ERR_ARG: return "a size or count is out of range";
        case SPEC_ERR_UNSUPPORTED: return "valid but unsupported shape or type";
        case SPEC_ERR_WORKSPACE: return "workspace missing or too small";
        case SPEC_ERR_CUDA: return "a CUDA runtime call failed";
        case SPEC_ERR_ALIGN: return "a pointer or row stride is not 16-byte aligned";
        default: return "unknown status";
    }
}

SPEC_API int spec_version(void) { return 200; }

namespace spec {
uint64_t g_wait_ns = DEFAULT_WAIT_NS;
}

SPEC_API void spec_test_set_wait_limit(uint64_t ns) { spec::g_wait_ns = ns ? ns : spec::DEFAULT_WAIT_NS; }
