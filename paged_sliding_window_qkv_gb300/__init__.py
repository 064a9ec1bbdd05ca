"""GB300-native paged two-family QKV prep + paged attention.

``pg`` is the ctypes binding of ``libpg.so`` (C ABI in ``include/pg.h``);
``runner`` sets up device buffers for one family; ``workloads`` draws seeded
synthetic inputs. Importing ``pg`` loads the native library and fails if it is
missing.
"""
