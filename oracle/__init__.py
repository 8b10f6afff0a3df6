"""CPU oracle for prefix-cached attention -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct implementations of what the GPU path computes, used to
check it.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import anything from here; the product path never does, and this
package never imports the product package (the two share no code).

Contents:
  attention.py / attention_ref.c  causal attention in fp64 over logical-order K/V
  radix_ref.py                    list matcher, dictionary model of the radix cache,
                                  seeded slot allocator, slot-table builder, shared-prefix groups
  merge.py                        combining softmax partial states over disjoint key sets
  toy_model.py                    random-weight causal LM for the cached-vs-full check

Every function is pinned by ``tests/test_oracle_*.py`` against closed forms,
invariants, brute force and the values the pages print.
"""
from .attention import attention_rows, build, max_threads  # noqa: F401
from .merge import merge_states  # noqa: F401
from .radix_ref import (ListMatcher, PrefixCacheModel, SlotAllocator, req_to_token,  # noqa: F401
                        shared_groups, slot_order, splitmix64)
