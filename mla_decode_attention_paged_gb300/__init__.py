"""Paged MLA decode attention for one GB300 (sm_103a): Python binding of the C-ABI library."""
