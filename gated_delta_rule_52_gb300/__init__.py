"""GB300-native (sm_103a) Kimi Delta Attention forward.

The product is the C-ABI library ``libkda.so`` (declared in ``include/kda.h``);
``gated_delta_rule_52_gb300.kda`` is its thin ctypes binding.  Importing this
package loads nothing; the library is opened on first use and a missing library
raises instead of falling back to any other implementation.
"""
