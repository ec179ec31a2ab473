"""Exact rational solver for integer systems A x = b by Dixon p-adic lifting,
GB300-native (sm_103a).  The compute path is the C-ABI library built from
``csrc/`` (declared in ``include/es.h``); this package is a thin binding."""
