// ddp_abi_guard.h -- no C++ exception leaves the library through its C ABI.
//
// The library's host code allocates with std::vector and std::map, which
// throw std::bad_alloc when host memory runs out.  An exception that unwinds
// into a C caller is undefined behaviour, so every status-returning entry
// point is a function-try-block ending in DDP_ABI_CATCH, which turns any
// exception into DDP_ERR_HOST.
#pragma once

#include "ddp.h"

#define DDP_ABI_CATCH \
    catch (...) {     \
        return DDP_ERR_HOST; \
    }
