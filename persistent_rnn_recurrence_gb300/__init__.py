"""Persistent ReLU-RNN recurrence for GB300 (sm_103a).

``synth`` draws seeded inputs; ``prnn`` is the thin ctypes binding of the C-ABI
library ``libprnn.so`` (built by ``persistent_rnn_recurrence_gb300.build``).
Importing the package loads nothing native; importing ``prnn`` does, and fails
loudly when the library is missing.
"""
