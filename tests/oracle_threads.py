"""Run the CPU oracle over token chunks on several host threads.

Test infrastructure: the oracle stays the plain single-threaded C code; this
helper only calls it on disjoint token ranges at once (ctypes releases the
GIL for the duration of each C call, and the oracle keeps no global state),
so that full-size workloads can be compared token by token in seconds."""
import concurrent.futures
import os

import oracle


def threads():
    return max(1, min(32, os.cpu_count() or 1))


def map_token_chunks(fn, T, chunk=4096):
    """fn(t0, t1) for every chunk [t0, t1) of [0, T), in parallel; results in
    token order."""
    oracle._load()  # build and load once, before the threads start
    ranges = [(t0, min(T, t0 + chunk)) for t0 in range(0, T, chunk)]
    with concurrent.futures.ThreadPoolExecutor(threads()) as ex:
        return list(ex.map(lambda r: fn(*r), ranges))
