// Library-internal queries on a handle (not part of the C ABI).
#pragma once

#include <stddef.h>

#include "../../include/blk.h"

__attribute__((visibility("hidden"))) size_t blk_internal_decode_ws_bytes(blk_handle h);
__attribute__((visibility("hidden"))) int blk_internal_device(blk_handle h);
