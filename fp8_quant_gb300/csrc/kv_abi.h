// The public C ABI, declared with default visibility: the library is built
// with -fvisibility=hidden, so only these entry points are exported.
#pragma once

#pragma GCC visibility push(default)
#include "kvstore.h"
#pragma GCC visibility pop
